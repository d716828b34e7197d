// Fused GEMV family for decode and small row counts (SIMT, f32 activations).
//
// One warp computes one output feature (or one gate/up pair) for up to ROWS
// activation rows; a CTA is 8 warps = 8 consecutive features; blockIdx.y is
// the row block. Each warp streams its weight row(s) with 128-bit loads issued
// before the activations are staged, so under programmatic dependent launch
// the weight fetch of this kernel overlaps the tail of the previous one.
//
// Prologue (QKV, SWIGLU, HEAD): RMSNorm of each activation row with the gain,
// x / sqrt(mean(x^2) + eps) * w ("qwentts.cpp/src/talker-forward.h",
// talker_layer_forward "Pre-norm" and the MLP pre-norm; talker_forward_core
// final norm). Epilogues: see talker_k::Epilogue.
#include <math.h>

#include "common.cuh"
#include "kernels.cuh"

using namespace talker_dev;

namespace talker_k {

// Index of element k of row r in the staged activation tile. For bf16
// weights a 16-byte weight vector covers 8 elements; its two halves are kept
// in two planes so that lane-consecutive vectors read contiguous float4s.
template <int EPV>
__device__ __forceinline__ int act_index(int r, int k, int K) {
    if (EPV == 8) return r * K + ((k >> 2) & 1) * (K >> 1) + (k >> 3) * 4 + (k & 3);
    return r * K + k;
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

__device__ __forceinline__ size_t cache_offset(const CacheView &c, int stream, int layer, int head, int pos) {
    const int page = c.page_table[stream * c.pages_per_stream + pos / kPage];
    return (size_t)page * c.page_elems + ((size_t)(layer * c.n_kv + head) * kPage + (pos % kPage)) * c.head_dim;
}

__device__ __forceinline__ int row_stream(const RowMap &m, int r) { return rowmap_stream(m, r); }
__device__ __forceinline__ int row_pos(const RowMap &m, int r) { return rowmap_pos(m, r); }

// QK-norm + NEOX RoPE + KV append for one completed head over the rows of a
// row block ("talker-forward.h", talker_layer_forward: per-head QK-norm, RoPE
// NEOX (half-split), set_rows into the cache at the fresh positions).
__device__ void finish_head(const GemvParams &p, int hidx, int row0, int nrows) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hd = p.head_dim, half = hd >> 1;
    const bool is_q = hidx < p.n_q;
    const bool is_k = !is_q && hidx < p.n_q + p.n_kv;
    const float *gain = is_q ? p.q_norm : p.k_norm;
    for (int r = warp; r < nrows; r += kGemvWarps) {
        const int row = row0 + r;
        const float *src = p.out + (size_t)row * p.out_ld + (size_t)hidx * hd;
        float a[2], b[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int i = lane + 32 * j;
            a[j] = (i < half) ? __ldcg(src + i) : 0.f;
            b[j] = (i < half) ? __ldcg(src + i + half) : 0.f;
        }
        const int pos = row_pos(p.rowmap, row);
        if (pos < 0 || pos >= p.cache.max_seq) {
            if (lane == 0) atomicOr(p.status, ST_BAD_POSITION);
            continue;
        }
        if (is_q || is_k) {
            float ss = a[0] * a[0] + b[0] * b[0] + a[1] * a[1] + b[1] * b[1];
            ss = warp_sum(ss);
            const float inv = 1.0f / sqrtf(ss / (float)hd + p.eps);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int i = lane + 32 * j;
                if (i < half) {
                    const float x0 = a[j] * inv * gain[i];
                    const float x1 = b[j] * inv * gain[i + half];
                    const float2 cs = p.rope[(size_t)pos * half + i];
                    a[j] = x0 * cs.x - x1 * cs.y;
                    b[j] = x1 * cs.x + x0 * cs.y;
                }
            }
        }
        if (is_q) {
            float *dst = p.q_out + (size_t)row * p.n_q * hd + (size_t)hidx * hd;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int i = lane + 32 * j;
                if (i < half) {
                    dst[i] = a[j];
                    dst[i + half] = b[j];
                }
            }
        } else {
            const int kvh = is_k ? hidx - p.n_q : hidx - p.n_q - p.n_kv;
            const int stream = row_stream(p.rowmap, row);
            const size_t off = cache_offset(p.cache, stream, p.layer, kvh, pos);
            void *base = is_k ? p.cache.k : p.cache.v;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int i = lane + 32 * j;
                if (i < half) {
                    if (p.cache.kv_bf16) {
                        __nv_bfloat16 *d = static_cast<__nv_bfloat16 *>(base) + off;
                        d[i] = __float2bfloat16_rn(a[j]);
                        d[i + half] = __float2bfloat16_rn(b[j]);
                    } else {
                        float *d = static_cast<float *>(base) + off;
                        d[i] = a[j];
                        d[i + half] = b[j];
                    }
                }
            }
        }
    }
}

__device__ __forceinline__ float4 ld_cluster_v4(const float *local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(remote)
                 : "memory");
    return v;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// EPI_SWIGLU_DOWN: CTAs whose down-projection partials are summed on chip, and the widest
// down output a CTA's threads cover (four outputs per thread).
constexpr int kFuseCluster = 8;
constexpr int kFuseMaxOut2 = 4 * kGemvThreads;

// VPL: 16-byte weight vectors a lane holds in flight per weight row (sized to K at
// launch, so that short rows leave registers free and more CTAs fit on an SM).
template <typename WT, int ROWS, int EPI, int VPL>
__global__ void __launch_bounds__(kGemvThreads) k_gemv(const GemvParams p) {
    constexpr int EPV = Elem<WT>::kPerVec;
    constexpr bool FUSED = (EPI == EPI_SWIGLU_DOWN);
    constexpr int NW = (EPI == EPI_SWIGLU || FUSED) ? 2 : 1;
    constexpr int MAXC = VPL;
    constexpr bool NORM = (EPI != EPI_RESID);
    extern __shared__ __align__(16) float act_s[];
    __shared__ float inv_s[ROWS];
    __shared__ float hv_s[kGemvWarps][ROWS];
    __shared__ int hi_s[kGemvWarps][ROWS];
    __shared__ int flag_s;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rb = blockIdx.y;
    const int row0 = rb * ROWS;
    const int nrows = min(ROWS, p.rows - row0);
    const int f = blockIdx.x * kGemvWarps + warp;
    const bool fvalid = f < p.n_out;
    const int K = p.K;
    const int nvec = K / EPV;
    const WT *wrow = static_cast<const WT *>(p.W) + (size_t)(NW * (fvalid ? f : 0)) * K;

    pdl_launch_dependents();

    // FUSED: this thread's down-projection weights W2[j][f0 .. f0 + 7] (j = tid + 256 i), 16 bytes
    // each; the cluster's 8 CTAs cover 128 contiguous bytes of every row j
    uint4 wd[FUSED ? 4 : 1];
    if constexpr (FUSED) {
        const int f0 = blockIdx.x * kGemvWarps;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int j = threadIdx.x + kGemvThreads * i;
            wd[i] = (j < p.n_out2) ? ldg_stream(static_cast<const __nv_bfloat16 *>(p.W2) + (size_t)j * p.n_out + f0)
                                   : make_uint4(0u, 0u, 0u, 0u);
        }
    }

    float acc[NW][ROWS];
#pragma unroll
    for (int n = 0; n < NW; ++n)
#pragma unroll
        for (int r = 0; r < ROWS; ++r) acc[n][r] = 0.f;
    float resid = 0.f;   // EPI_RESID: this lane's residual value, fetched right after the wait

    for (int base = 0; base < nvec; base += 32 * MAXC) {
        uint4 w[NW][MAXC];
#pragma unroll
        for (int n = 0; n < NW; ++n)
#pragma unroll
            for (int i = 0; i < MAXC; ++i) {
                const int c = base + i * 32 + lane;
                w[n][i] = (fvalid && c < nvec) ? ldg_stream(wrow + (size_t)n * K + (size_t)c * EPV)
                                               : make_uint4(0u, 0u, 0u, 0u);
            }
        if (base == 0) {
            // Activations are produced by the previous kernel: wait for it only now. All
            // threads stage the rows (one round trip), then the RMSNorm is reduced from
            // shared memory and applied in place.
            pdl_wait();
            if (EPI == EPI_RESID && lane < nrows && fvalid) resid = p.out[(size_t)(row0 + lane) * p.out_ld + f];
            const int K4 = K >> 2;
            const bool do_copy = (p.copy_x != nullptr) && blockIdx.x == 0;
            float ss[ROWS];
#pragma unroll
            for (int r = 0; r < ROWS; ++r) ss[r] = 0.f;
            for (int idx = threadIdx.x; idx < nrows * K4; idx += kGemvThreads) {
                const int r = idx / K4, k = (idx - r * K4) * 4;
                float4 v;
                if (EPI == EPI_QKV && p.gather.n > 0)   // only the first layer's QKV projection gathers
                    v = gather_row4(p.gather, row0 + r, k, K, p.status);
                else
                    v = *reinterpret_cast<const float4 *>(p.act + (size_t)(row0 + r) * p.act_ld + k);
                if (do_copy) *reinterpret_cast<float4 *>(p.copy_x + (size_t)(row0 + r) * K + k) = v;
                *reinterpret_cast<float4 *>(act_s + act_index<EPV>(r, k, K)) = v;
                if (NORM) {
                    const float q = v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
#pragma unroll
                    for (int rr = 0; rr < ROWS; ++rr)
                        if (rr == r) ss[rr] += q;
                }
            }
            if (NORM) {
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    const float t = warp_sum(ss[r]);
                    if (lane == 0) hv_s[warp][r] = t;
                }
                __syncthreads();
                if (threadIdx.x < nrows) {
                    float t = 0.f;
                    for (int w = 0; w < kGemvWarps; ++w) t += hv_s[w][threadIdx.x];
                    inv_s[threadIdx.x] = 1.0f / sqrtf(t / (float)K + p.eps);
                }
                __syncthreads();
                for (int idx = threadIdx.x; idx < nrows * K4; idx += kGemvThreads) {
                    const int r = idx / K4, k = (idx - r * K4) * 4;
                    float4 *a = reinterpret_cast<float4 *>(act_s + act_index<EPV>(r, k, K));
                    const float4 g = *reinterpret_cast<const float4 *>(p.norm_w + k);
                    float4 v = *a;
                    const float iv = inv_s[r];
                    v.x = v.x * iv * g.x;
                    v.y = v.y * iv * g.y;
                    v.z = v.z * iv * g.z;
                    v.w = v.w * iv * g.w;
                    *a = v;
                }
            }
            __syncthreads();
        }
#pragma unroll
        for (int i = 0; i < MAXC; ++i) {
            const int c = base + i * 32 + lane;
            if (c < nvec) {
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    if (r < nrows) {
                        if (EPV == 8) {
                            const float4 a0 = *reinterpret_cast<const float4 *>(act_s + r * K + c * 4);
                            const float4 a1 = *reinterpret_cast<const float4 *>(act_s + r * K + (K >> 1) + c * 4);
#pragma unroll
                            for (int n = 0; n < NW; ++n) {
                                const uint4 u = w[n][i];
                                float s = acc[n][r];
                                s = fmaf(bf16lo(u.x), a0.x, s);
                                s = fmaf(bf16hi(u.x), a0.y, s);
                                s = fmaf(bf16lo(u.y), a0.z, s);
                                s = fmaf(bf16hi(u.y), a0.w, s);
                                s = fmaf(bf16lo(u.z), a1.x, s);
                                s = fmaf(bf16hi(u.z), a1.y, s);
                                s = fmaf(bf16lo(u.w), a1.z, s);
                                s = fmaf(bf16hi(u.w), a1.w, s);
                                acc[n][r] = s;
                            }
                        } else {
                            const float4 a0 = *reinterpret_cast<const float4 *>(act_s + r * K + c * 4);
#pragma unroll
                            for (int n = 0; n < NW; ++n) {
                                const uint4 u = w[n][i];
                                float s = acc[n][r];
                                s = fmaf(__uint_as_float(u.x), a0.x, s);
                                s = fmaf(__uint_as_float(u.y), a0.y, s);
                                s = fmaf(__uint_as_float(u.z), a0.z, s);
                                s = fmaf(__uint_as_float(u.w), a0.w, s);
                                acc[n][r] = s;
                            }
                        }
                    }
                }
            }
        }
    }

    // ---- epilogue
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        float v0 = warp_sum(acc[0][r]);
        const float v1 = (NW == 2) ? warp_sum(acc[NW - 1][r]) : 0.f;
        if (EPI == EPI_HEAD && p.suppress_tail > 0 && f >= p.n_out - p.suppress_tail && f != p.eos_id)
            v0 = -INFINITY;   // codebook-0 suppression of the vocabulary tail (EOS kept)
        if (EPI == EPI_HEAD && lane == r) {
            hv_s[warp][r] = (fvalid && r < nrows) ? v0 : -INFINITY;
            hi_s[warp][r] = f;
        }
        if (FUSED) {
            if (lane == r) hv_s[warp][r] = (r < nrows && fvalid) ? silu_f(v0) * v1 : 0.f;
        } else if (lane == r && r < nrows && fvalid) {
            float *o = p.out + (size_t)(row0 + r) * p.out_ld + f;
            if (EPI == EPI_RESID) {
                *o = resid + v0;
                if (p.out2 != nullptr) p.out2[(size_t)(row0 + r) * p.out_ld + f] = resid + v0;
            } else if (EPI == EPI_SWIGLU) {
                *o = silu_f(v0) * v1;
            } else {
                *o = v0;
            }
        }
    }

    if constexpr (FUSED) {
        // partial down products of this CTA's 8 activations a[f0 .. f0 + 7] for every output j
        // ("talker-forward.h", talker_layer_forward MLP: down(silu(gate) * up)), kept in shared
        // memory; the cluster's 8 CTAs then sum them (rank k owns outputs [k n2/8, (k+1) n2/8))
        // and reduce-add the sums into red_out, which holds the residual stream
        __syncthreads();
        const int n2 = p.n_out2;
        float *part_s = act_s + ROWS * K;   // [ROWS][n2]
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            if (r < nrows) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int j = threadIdx.x + kGemvThreads * i;
                    if (j < n2) {
                        const uint4 u = wd[i];
                        float t = bf16lo(u.x) * hv_s[0][r];
                        t = fmaf(bf16hi(u.x), hv_s[1][r], t);
                        t = fmaf(bf16lo(u.y), hv_s[2][r], t);
                        t = fmaf(bf16hi(u.y), hv_s[3][r], t);
                        t = fmaf(bf16lo(u.z), hv_s[4][r], t);
                        t = fmaf(bf16hi(u.z), hv_s[5][r], t);
                        t = fmaf(bf16lo(u.w), hv_s[6][r], t);
                        t = fmaf(bf16hi(u.w), hv_s[7][r], t);
                        part_s[r * n2 + j] = t;
                    }
                }
            }
        }
        cluster_sync_all();
        uint32_t rank;
        asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
        const int per = n2 / kFuseCluster, per4 = per / 4;
        for (int idx = threadIdx.x; idx < nrows * per4; idx += kGemvThreads) {
            const int r = idx / per4, j = (int)rank * per + (idx - r * per4) * 4;
            float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int c = 0; c < kFuseCluster; ++c) {
                const float4 v = ld_cluster_v4(part_s + r * n2 + j, (uint32_t)c);
                t.x += v.x;
                t.y += v.y;
                t.z += v.z;
                t.w += v.w;
            }
            float *o = p.red_out + (size_t)(row0 + r) * n2 + j;
            asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(o), "f"(t.x), "f"(t.y), "f"(t.z),
                         "f"(t.w)
                         : "memory");
        }
        cluster_sync_all();   // peers read this CTA's partials: keep its shared memory until they are done
    }

    if (EPI == EPI_QKV && p.q_out != nullptr) {
        __threadfence();
        __syncthreads();
        const int hidx = (blockIdx.x * kGemvWarps) / p.head_dim;
        const int n_heads = p.n_q + 2 * p.n_kv;
        int *cnt = p.cnt + (size_t)rb * n_heads + hidx;
        if (threadIdx.x == 0) {
            __threadfence();
            const int old = atomicAdd(cnt, 1);
            flag_s = (old == p.head_dim / kGemvWarps - 1);
        }
        __syncthreads();
        if (flag_s) {
            __threadfence();
            finish_head(p, hidx, row0, nrows);
            if (threadIdx.x == 0) *cnt = 0;
        }
    }

    if (EPI == EPI_HEAD) {
        __syncthreads();
        if (p.hidden_out != nullptr && blockIdx.x == 0) {
            for (int idx = threadIdx.x; idx < nrows * K; idx += kGemvThreads) {
                const int r = idx / K, k = idx - r * K;
                p.hidden_out[(size_t)(row0 + r) * K + k] = act_s[act_index<EPV>(r, k, K)];
            }
        }
        if (threadIdx.x < nrows) {
            const int r = threadIdx.x;
            float best = -INFINITY;
            int bi = 0x7fffffff;
            for (int w = 0; w < kGemvWarps; ++w) {
                float v = hv_s[w][r];
                const int i = hi_s[w][r];
                if (isnan(v)) {   // reported, and ranked as -inf: the argmax stays a valid index
                    atomicOr(p.status, ST_NAN_LOGIT);
                    v = -INFINITY;
                }
                if (v > best || (v == best && i < bi)) {
                    best = v;
                    bi = i;
                }
            }
            const size_t slot = ((size_t)rb * gridDim.x + blockIdx.x) * ROWS + r;
            p.part_val[slot] = best;
            p.part_idx[slot] = bi;
        }
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            const int old = atomicAdd(p.head_cnt + rb, 1);
            flag_s = (old == (int)gridDim.x - 1);
        }
        __syncthreads();
        if (flag_s) {
            __threadfence();
            // the last CTA reduces the per-CTA partials: one warp per row (rows spread over the
            // warps, every lane's loads in flight together), lowest index on ties
            for (int r = warp; r < nrows; r += kGemvWarps) {
                float best = -INFINITY;
                int bi = 0x7fffffff;
#pragma unroll 4
                for (int b = lane; b < (int)gridDim.x; b += 32) {
                    const size_t slot = ((size_t)rb * gridDim.x + b) * ROWS + r;
                    const float v = __ldcg(p.part_val + slot);
                    const int i = __ldcg(p.part_idx + slot);
                    if (v > best || (v == best && i < bi)) {
                        best = v;
                        bi = i;
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float v2 = __shfl_xor_sync(0xffffffffu, best, o);
                    const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
                    if (v2 > best || (v2 == best && i2 < bi)) {
                        best = v2;
                        bi = i2;
                    }
                }
                if (lane == 0) {
                    if (p.argmax_out != nullptr) p.argmax_out[row0 + r] = bi;
                    if (p.inc_len) p.cur_len_rw[row0 + r] += 1;
                }
            }
            __syncthreads();
            if (threadIdx.x == 0) p.head_cnt[rb] = 0;
        }
    }
}

int gemv_rows_for(int rows) { return rows <= 1 ? 1 : (rows <= 4 ? 4 : 16); }

size_t gemv_smem_bytes(int rows_tmpl, int K) { return (size_t)rows_tmpl * K * sizeof(float); }

template <typename WT, int ROWS, int EPI, int VPL>
static cudaError_t launch_vpl(const GemvParams &p, cudaStream_t st, bool pdl) {
    const int nfeat = p.n_out;
    dim3 grid((nfeat + kGemvWarps - 1) / kGemvWarps, (p.rows + ROWS - 1) / ROWS, 1);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kGemvThreads, 1, 1);
    cfg.dynamicSmemBytes = gemv_smem_bytes(ROWS, p.K);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (EPI == EPI_SWIGLU_DOWN) {
        if (grid.x % kFuseCluster || p.n_out % kGemvWarps || p.n_out2 % (4 * kFuseCluster) ||
            p.n_out2 > kFuseMaxOut2 || p.W2 == nullptr || p.red_out == nullptr)
            return cudaErrorInvalidValue;
        cfg.dynamicSmemBytes += (size_t)ROWS * p.n_out2 * sizeof(float);
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = kFuseCluster;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, k_gemv<WT, ROWS, EPI, VPL>, p);
}

// Vectors per lane of one weight row, rounded up to an instantiated size.
template <typename WT>
static int vpl_for(int K) {
    const int v = (K / Elem<WT>::kPerVec + 31) / 32;
    return v <= 4 ? 4 : (v <= 8 ? 8 : 16);
}

template <typename WT, int ROWS, int EPI>
static cudaError_t launch_one(const GemvParams &p, cudaStream_t st, bool pdl) {
    switch (vpl_for<WT>(p.K)) {
        case 4: return launch_vpl<WT, ROWS, EPI, 4>(p, st, pdl);
        case 8: return launch_vpl<WT, ROWS, EPI, 8>(p, st, pdl);
    }
    return launch_vpl<WT, ROWS, EPI, 16>(p, st, pdl);
}

template <typename WT, int ROWS>
static cudaError_t launch_rows(int epi, const GemvParams &p, cudaStream_t st, bool pdl) {
    switch (epi) {
        case EPI_QKV: return launch_one<WT, ROWS, EPI_QKV>(p, st, pdl);
        case EPI_RESID: return launch_one<WT, ROWS, EPI_RESID>(p, st, pdl);
        case EPI_SWIGLU: return launch_one<WT, ROWS, EPI_SWIGLU>(p, st, pdl);
        case EPI_HEAD: return launch_one<WT, ROWS, EPI_HEAD>(p, st, pdl);
        case EPI_SWIGLU_DOWN:
            if constexpr (sizeof(WT) == 2) return launch_one<WT, ROWS, EPI_SWIGLU_DOWN>(p, st, pdl);
            return cudaErrorInvalidValue;
    }
    return cudaErrorInvalidValue;
}

template <typename WT>
static cudaError_t launch_wt(int epi, int rows_tmpl, const GemvParams &p, cudaStream_t st, bool pdl) {
    switch (rows_tmpl) {
        case 1: return launch_rows<WT, 1>(epi, p, st, pdl);
        case 4: return launch_rows<WT, 4>(epi, p, st, pdl);
        case 16: return launch_rows<WT, 16>(epi, p, st, pdl);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_gemv(int epi, int w_bf16, int rows_tmpl, const GemvParams &p, cudaStream_t st, bool pdl) {
    if (w_bf16) return launch_wt<__nv_bfloat16>(epi, rows_tmpl, p, st, pdl);
    return launch_wt<float>(epi, rows_tmpl, p, st, pdl);
}

template <typename WT, int ROWS, int VPL>
static cudaError_t raise_vpl() {
    const int bytes = 200 * 1024;
    cudaError_t e = cudaSuccess;
    e = e ? e : cudaFuncSetAttribute(k_gemv<WT, ROWS, EPI_QKV, VPL>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    e = e ? e : cudaFuncSetAttribute(k_gemv<WT, ROWS, EPI_RESID, VPL>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    e = e ? e : cudaFuncSetAttribute(k_gemv<WT, ROWS, EPI_SWIGLU, VPL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     bytes);
    e = e ? e : cudaFuncSetAttribute(k_gemv<WT, ROWS, EPI_HEAD, VPL>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if constexpr (sizeof(WT) == 2)
        e = e ? e : cudaFuncSetAttribute(k_gemv<WT, ROWS, EPI_SWIGLU_DOWN, VPL>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    return e;
}

template <typename WT, int ROWS>
static cudaError_t raise_rows() {
    cudaError_t e = raise_vpl<WT, ROWS, 4>();
    e = e ? e : raise_vpl<WT, ROWS, 8>();
    return e ? e : raise_vpl<WT, ROWS, 16>();
}

cudaError_t prepare_gemv() {
    cudaError_t e = cudaSuccess;
    e = e ? e : raise_rows<float, 1>();
    e = e ? e : raise_rows<float, 4>();
    e = e ? e : raise_rows<float, 16>();
    e = e ? e : raise_rows<__nv_bfloat16, 1>();
    e = e ? e : raise_rows<__nv_bfloat16, 4>();
    e = e ? e : raise_rows<__nv_bfloat16, 16>();
    return e;
}

}  // namespace talker_k
