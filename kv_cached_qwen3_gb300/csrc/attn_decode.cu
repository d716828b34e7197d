// Split-K flash-decode GQA attention over the paged KV cache.
//
// Computes, for each query row r (stream s, position p) and q head h,
//   o_h = softmax_j(q_h . k_{g,j} / sqrt(hd)) v_{g,j},  j in [0, p],  g = h / (n_q / n_kv)
// ("qwentts.cpp/src/talker-forward.h", talker_layer_forward: flash_attn_ext
// with F32 precision over the causal window; GQA by repeat_interleave of the KV
// heads as in "causal_lm.cpp"). The window is bounded by the row's length, not
// by a mask, so cache rows past p are never read into the arithmetic.
//
// Grid (splits, n_kv, rows). CTA (split, g, r) walks a contiguous range of
// 64-position pages of (s, layer, g); each K and V page tile is one contiguous
// block moved into shared memory by a bulk (TMA) copy, double buffered. All
// q heads of the group share each tile. Running max / sum / output are fp32
// (online softmax). Each CTA writes its partial (m, l, o); the CTA that
// finishes last for (r, g) (atomic counter, no waiting) combines the partials
// in split order, so the result is deterministic.
#include <math.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.cuh"

using namespace talker_dev;

namespace talker_k {

constexpr int kMaxGroup = 8;

__device__ __forceinline__ int attn_row_stream(const RowMap &m, int r) { return rowmap_stream(m, r); }
__device__ __forceinline__ int attn_row_pos(const RowMap &m, int r) {
    return rowmap_pos(m, r);
}

// One (page, layer, KV head) tile of the cache as it sits in the pool and in shared memory.
// bf16 / f32: [64][HD] values. Q8_0 (KT = int8_t): [64][HD] codes, then [64][HD/32] fp16 scales.
template <typename KT, int HD>
struct KvTile {
    static constexpr uint32_t kBytes = kPage * HD * sizeof(KT);
    static constexpr size_t kUnits = (size_t)kPage * HD;   // pool units (elements) per tile
    __device__ static __forceinline__ float load(const unsigned char *t, int j, int d) {
        return Elem<KT>::load(reinterpret_cast<const KT *>(t), (size_t)j * HD + d);
    }
};
template <int HD>
struct KvTile<int8_t, HD> {   // int8 stands for the Q8_0 storage type
    static constexpr uint32_t kBytes = kPage * HD + kPage * (HD / 32) * 2;
    static constexpr size_t kUnits = kBytes;                // pool units are bytes
    __device__ static __forceinline__ float load(const unsigned char *t, int j, int d) {
        const float c = (float)reinterpret_cast<const int8_t *>(t)[j * HD + d];
        return c * __half2float(reinterpret_cast<const __half *>(t + kPage * HD)[j * (HD / 32) + (d >> 5)]);
    }
};

size_t attn_smem_bytes(int kv_kind, int head_dim, int group) {
    // kv_kind: 0 f32, 1 bf16, 2 Q8_0
    const size_t tile = kv_kind == 2 ? (size_t)kPage * head_dim + (size_t)kPage * (head_dim / 32) * 2
                                     : (size_t)kPage * head_dim * (kv_kind == 1 ? 2 : 4);
    return 4 * tile + (size_t)group * head_dim * 4 + (size_t)group * kPage * 4 + 2 * (size_t)head_dim * 4;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float ld_cluster_f32(const void *local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

// Combination of the splits of one (row, KV group) when they form one thread-block
// cluster: every CTA leaves its (m, l, o) in its own shared memory (o_part, m_part,
// l_part; an empty split has m = -inf), the cluster synchronises, CTA rank 0 reads the
// partials of all ranks through distributed shared memory in rank order and writes the
// output row, and a second cluster barrier keeps every CTA (and its shared memory) alive
// until rank 0 is done. Every CTA of the cluster calls this exactly once.
template <int HD>
__device__ void cluster_combine(const AttnParams &p, bool has, const float *o_part, float *m_part, float *l_part,
                                int r, int g) {
    const int G = p.group, tid = threadIdx.x;
    if (!has && tid < G) {
        m_part[tid] = -INFINITY;
        l_part[tid] = 0.f;
    }
    __syncthreads();
    cluster_sync_all();
    uint32_t rank, nranks;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(nranks));
    if (rank == 0) {
        const size_t out_row = (size_t)r * p.n_q * HD;
        for (int idx = tid; idx < G * HD; idx += kAttnThreads) {
            const int gi = idx / HD, d = idx - gi * HD;
            float M = -INFINITY;
            for (uint32_t c = 0; c < nranks; ++c) M = fmaxf(M, ld_cluster_f32(m_part + gi, c));
            float L = 0.f, O = 0.f;
            for (uint32_t c = 0; c < nranks; ++c) {
                const float mc = ld_cluster_f32(m_part + gi, c);
                if (mc == -INFINITY) continue;
                const float f = expf(mc - M);
                L = fmaf(ld_cluster_f32(l_part + gi, c), f, L);
                O = fmaf(ld_cluster_f32(o_part + idx, c), f, O);
            }
            const float v = O / L;
            const size_t oi = out_row + (size_t)(g * G + gi) * HD + d;
            if (p.out_bf16) static_cast<__nv_bfloat16 *>(p.out)[oi] = __float2bfloat16_rn(v);
            else static_cast<float *>(p.out)[oi] = v;
        }
    }
    cluster_sync_all();
}

template <typename KT, int HD>
__global__ void __launch_bounds__(kAttnThreads) k_attn_decode(const AttnParams p) {
    using Tile = KvTile<KT, HD>;
    constexpr bool kQ8 = std::is_same<KT, int8_t>::value;
    constexpr int E = HD / 32;                       // elements of a key row per lane
    constexpr int NO = (kMaxGroup * HD + kAttnThreads - 1) / kAttnThreads;
    constexpr uint32_t kTileBytes = Tile::kBytes;
    constexpr size_t kUnit = kQ8 ? 1 : sizeof(KT);   // bytes per pool unit
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *kbuf = smem_raw;                                      // [2][tile]
    unsigned char *vbuf = kbuf + 2 * kTileBytes;                         // [2][tile]
    float *q_s = reinterpret_cast<float *>(vbuf + 2 * kTileBytes);       // [G][HD]
    float *sc = q_s + p.group * HD;                                      // [G][kPage]
    float *knew = sc + p.group * kPage;                                  // this step's k, v row (as attended)
    float *vnew = knew + HD;
    __shared__ float m_s[kMaxGroup], l_s[kMaxGroup], al_s[kMaxGroup];
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ int flag_s;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int sidx = blockIdx.x, g = blockIdx.y, r = blockIdx.z;
    const int G = p.group;

    pdl_launch_dependents();
    // Decode rows: before the wait on the previous kernel (which writes q and this step's
    // k / v row) only data of earlier launches is read: the length, the page table and the
    // cached pages. The page holding position pos is patched with the fresh row after the
    // wait. Prefill rows (all of them fresh) wait first.
    if (p.rowmap.mode != 0) pdl_wait();

    const int s = attn_row_stream(p.rowmap, r);
    const int pos = attn_row_pos(p.rowmap, r);
    if (pos < 0 || pos >= p.cache.max_seq) {
        if (tid == 0 && sidx == 0) atomicOr(p.status, ST_BAD_POSITION);
        return;
    }
    const int nvis = pos + 1;
    const int npages = (nvis + kPage - 1) / kPage;
    const int per = (npages + p.splits - 1) / p.splits;
    const int pb = sidx * per;
    const int pe = min(pb + per, npages);
    const int nact = (npages + per - 1) / per;
    if (pb >= pe) {   // no pages for this split
        if (p.cluster && nact > 1) cluster_combine<HD>(p, false, q_s, m_s, l_s, r, g);
        return;
    }

    const int *ptab = p.cache.page_table + (size_t)s * p.cache.pages_per_stream;
    const size_t head_off = (size_t)(p.layer * p.cache.n_kv + g) * Tile::kUnits;   // pool units
    const unsigned char *kpool = static_cast<const unsigned char *>(p.cache.k);
    const unsigned char *vpool = static_cast<const unsigned char *>(p.cache.v);
    auto tile_ptr = [&](const unsigned char *pool, int page) {
        return pool + ((size_t)page * p.cache.page_elems + head_off) * kUnit;
    };

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (tid == 0) {
        mbar_arrive_expect_tx(&bars[0], 2 * kTileBytes);
        bulk_g2s(kbuf, tile_ptr(kpool, ptab[pb]), kTileBytes, &bars[0]);
        bulk_g2s(vbuf, tile_ptr(vpool, ptab[pb]), kTileBytes, &bars[0]);
    }
    // the RoPE row of this position (a table of earlier launches) is fetched before the wait
    constexpr int half_hd = HD / 2;
    float2 cs_pre[2] = {make_float2(1.f, 0.f), make_float2(1.f, 0.f)};
    if (p.raw != nullptr && warp <= G) {
#pragma unroll
        for (int j = 0; j < 2; ++j)
            if (lane + 32 * j < half_hd) cs_pre[j] = p.rope[(size_t)pos * half_hd + lane + 32 * j];
    }
    pdl_wait();
    if (p.raw == nullptr) {
        const float *qsrc = p.q + (size_t)r * p.n_q * HD + (size_t)g * G * HD;
        for (int i = tid; i < G * HD; i += kAttnThreads) q_s[i] = qsrc[i] * p.scale;
    } else {
        // heads of this group from the raw projections: q heads g*G.., k head g, v head g;
        // QK-norm and RoPE ("talker-forward.h", talker_layer_forward), k / v appended by split 0
        constexpr int half = HD / 2;
        for (int hh = warp; hh < G + 2; hh += kAttnThreads / 32) {
            const int hidx = hh < G ? g * G + hh : (hh == G ? p.n_q + g : p.n_q + p.n_kv + g);
            const float *src = p.raw + (size_t)r * p.qkv_n + (size_t)hidx * HD;
            float a[2], b[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int i = lane + 32 * j;
                a[j] = (i < half) ? src[i] : 0.f;
                b[j] = (i < half) ? src[i + half] : 0.f;
            }
            if (hh <= G) {
                const float *gain = hh < G ? p.q_norm : p.k_norm;
                const float ss = warp_sum(a[0] * a[0] + b[0] * b[0] + a[1] * a[1] + b[1] * b[1]);
                const float inv = 1.0f / sqrtf(ss / (float)HD + p.eps);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int i = lane + 32 * j;
                    if (i < half) {
                        const float x0 = a[j] * inv * gain[i], x1 = b[j] * inv * gain[i + half];
                        const float2 cs = (hh == warp) ? cs_pre[j] : p.rope[(size_t)pos * half + i];
                        a[j] = x0 * cs.x - x1 * cs.y;
                        b[j] = x1 * cs.x + x0 * cs.y;
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int i = lane + 32 * j;
                if (i >= half) continue;
                if (hh < G) {
                    q_s[hh * HD + i] = a[j] * p.scale;
                    q_s[hh * HD + i + half] = b[j] * p.scale;
                } else {
                    // the row as this step attends it: exact with Q8_0 storage, else as stored
                    float *d = hh == G ? knew : vnew;
                    if constexpr (kQ8) {
                        d[i] = a[j];
                        d[i + half] = b[j];
                    } else {
                        d[i] = Elem<KT>::round(a[j]);
                        d[i + half] = Elem<KT>::round(b[j]);
                        if (sidx == 0) {   // the cache keeps the row for later steps
                            unsigned char *t =
                                const_cast<unsigned char *>(tile_ptr(hh == G ? kpool : vpool, ptab[pos / kPage]));
                            KT *c = reinterpret_cast<KT *>(t) + (size_t)(pos % kPage) * HD;
                            Elem<KT>::store(c, i, a[j]);
                            Elem<KT>::store(c, i + half, b[j]);
                        }
                    }
                }
            }
            if (kQ8 && hh >= G && sidx == 0) {
                // Q8_0 row: each valid register of the warp is one block of 32 dims (lane = dim % 32)
                unsigned char *t = const_cast<unsigned char *>(tile_ptr(hh == G ? kpool : vpool, ptab[pos / kPage]));
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int d0 = 32 * j + u * half;   // first dim of this register's block
                        if (32 * j >= half) continue;
                        q8_store_block(t, (pos % kPage) * HD + d0, kPage * HD + ((pos % kPage) * (HD / 32) + d0 / 32) * 2,
                                       u ? b[j] : a[j], lane);
                    }
            }
        }
    }
    if (tid < G) {
        m_s[tid] = -INFINITY;
        l_s[tid] = 0.f;
    }
    float o_acc[NO];
#pragma unroll
    for (int o = 0; o < NO; ++o) o_acc[o] = 0.f;
    __syncthreads();

    bool failed = false;
    int fail_it = 0;
    for (int pg = pb, it = 0; pg < pe; ++pg, ++it) {
        const int buf = it & 1;
        const uint32_t parity = (it >> 1) & 1;
        if (tid == 0 && pg + 1 < pe) {
            // The other buffer was released by the barrier that ended the previous iteration.
            fence_proxy_async();
            mbar_arrive_expect_tx(&bars[buf ^ 1], 2 * kTileBytes);
            bulk_g2s(kbuf + (buf ^ 1) * kTileBytes, tile_ptr(kpool, ptab[pg + 1]), kTileBytes, &bars[buf ^ 1]);
            bulk_g2s(vbuf + (buf ^ 1) * kTileBytes, tile_ptr(vpool, ptab[pg + 1]), kTileBytes, &bars[buf ^ 1]);
        }
        const bool ok = mbar_wait(&bars[buf], parity, p.status);
        if (__syncthreads_or(!ok)) {
            failed = true;
            fail_it = it;
            break;
        }
        const unsigned char *Ks = kbuf + buf * kTileBytes;
        const unsigned char *Vs = vbuf + buf * kTileBytes;
        const int valid = min(kPage, nvis - pg * kPage);
        // decode rows: row `newest` of this page is this step's row, read from knew / vnew (the
        // copied page may predate it); prefill rows were all written before the page was copied
        const int newest = (p.raw != nullptr) ? pos - pg * kPage : -1;
        if constexpr (!kQ8) {   // bf16 / f32 tiles hold the fresh row exactly as stored: patch it in
            if (newest >= 0 && newest < kPage) {
                KT *kt = reinterpret_cast<KT *>(kbuf + buf * kTileBytes) + newest * HD;
                KT *vt = reinterpret_cast<KT *>(vbuf + buf * kTileBytes) + newest * HD;
                for (int i = tid; i < HD; i += kAttnThreads) {
                    Elem<KT>::store(kt, i, knew[i]);
                    Elem<KT>::store(vt, i, vnew[i]);
                }
                __syncthreads();
            }
        }

        // scores: warp w takes key rows w, w + 8, ...; lanes split the head dimension. All of a
        // warp's rows and heads are reduced in one interleaved butterfly (latency paid once).
        {
            constexpr int NWARP = kAttnThreads / 32;
            constexpr int RPW = kPage / NWARP;   // rows per warp
            float kv[RPW][E];
#pragma unroll
            for (int i = 0; i < RPW; ++i)
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const int j = warp + NWARP * i;
                    if constexpr (kQ8) kv[i][e] = (j == newest) ? knew[lane * E + e] : Tile::load(Ks, j, lane * E + e);
                    else kv[i][e] = Tile::load(Ks, j, lane * E + e);
                }
            for (int gi0 = 0; gi0 < G; gi0 += 2) {   // two heads per pass keeps the register count bounded
                float dv[RPW][2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int gi = min(gi0 + u, G - 1);
                    float qv[E];
#pragma unroll
                    for (int e = 0; e < E; ++e) qv[e] = q_s[gi * HD + lane * E + e];
#pragma unroll
                    for (int i = 0; i < RPW; ++i) {
                        float d = 0.f;
#pragma unroll
                        for (int e = 0; e < E; ++e) d = fmaf(qv[e], kv[i][e], d);
                        dv[i][u] = d;
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                    for (int i = 0; i < RPW; ++i) {
                        dv[i][0] += __shfl_xor_sync(0xffffffffu, dv[i][0], o);
                        dv[i][1] += __shfl_xor_sync(0xffffffffu, dv[i][1], o);
                    }
                if (lane == 0) {
#pragma unroll
                    for (int i = 0; i < RPW; ++i) {
                        const int j = warp + NWARP * i;
                        sc[gi0 * kPage + j] = (j < valid) ? dv[i][0] : -INFINITY;
                        if (gi0 + 1 < G) sc[(gi0 + 1) * kPage + j] = (j < valid) ? dv[i][1] : -INFINITY;
                    }
                }
            }
        }
        __syncthreads();
        // online softmax update, one warp per q head of the group
        if (warp < G) {
            const int gi = warp;
            const float v0 = sc[gi * kPage + lane], v1 = sc[gi * kPage + lane + 32];
            const float mp = warp_max(fmaxf(v0, v1));
            const float m_old = m_s[gi];
            const float m_new = fmaxf(m_old, mp);
            const float alpha = expf(m_old - m_new);
            const float p0 = (lane < valid) ? expf(v0 - m_new) : 0.f;
            const float p1 = (lane + 32 < valid) ? expf(v1 - m_new) : 0.f;
            sc[gi * kPage + lane] = p0;
            sc[gi * kPage + lane + 32] = p1;
            const float ls = warp_sum(p0 + p1);
            if (lane == 0) {
                l_s[gi] = l_s[gi] * alpha + ls;
                m_s[gi] = m_new;
                al_s[gi] = alpha;
            }
        }
        __syncthreads();
        // o = o * alpha + sum_j p_j v_j over the valid rows only
#pragma unroll
        for (int o = 0; o < NO; ++o) {
            const int idx = tid + o * kAttnThreads;
            if (idx < G * HD) {
                const int gi = idx / HD, d = idx - gi * HD;
                // four independent chains over the page's rows
                float a0 = o_acc[o] * al_s[gi], a1 = 0.f, a2 = 0.f, a3 = 0.f;
                const float *pj = sc + gi * kPage;
                // the fresh row, when this page holds it, is the page's last valid row: it is
                // added from vnew after the branch-free loop over the copied rows
                const int vmain = (newest >= 0 && newest < valid) ? valid - 1 : valid;
                int j = 0;
                for (; j + 4 <= vmain; j += 4) {
                    a0 = fmaf(pj[j], Tile::load(Vs, j, d), a0);
                    a1 = fmaf(pj[j + 1], Tile::load(Vs, j + 1, d), a1);
                    a2 = fmaf(pj[j + 2], Tile::load(Vs, j + 2, d), a2);
                    a3 = fmaf(pj[j + 3], Tile::load(Vs, j + 3, d), a3);
                }
                for (; j < vmain; ++j) a0 = fmaf(pj[j], Tile::load(Vs, j, d), a0);
                if (vmain < valid) a0 = fmaf(pj[vmain], vnew[d], a0);
                o_acc[o] = (a0 + a1) + (a2 + a3);
            }
        }
        __syncthreads();
    }
    if (failed) {
        // Give the copies still in flight (this page's, and the next page's if it
        // was prefetched) a bounded chance to land before the CTA exits.
        if (tid == 0) {
            mbar_wait(&bars[fail_it & 1], (fail_it >> 1) & 1, p.status);
            if (pb + fail_it + 1 < pe) mbar_wait(&bars[(fail_it + 1) & 1], ((fail_it + 1) >> 1) & 1, p.status);
        }
        __syncthreads();
        if (p.cluster && nact > 1) cluster_combine<HD>(p, false, q_s, m_s, l_s, r, g);
        return;
    }

    const int hq0 = g * G;
    const size_t out_row = (size_t)r * p.n_q * HD;
    if (nact == 1) {
#pragma unroll
        for (int o = 0; o < NO; ++o) {
            const int idx = tid + o * kAttnThreads;
            if (idx < G * HD) {
                const int gi = idx / HD, d = idx - gi * HD;
                const float v = o_acc[o] / l_s[gi];
                const size_t oi = out_row + (size_t)(hq0 + gi) * HD + d;
                if (p.out_bf16) static_cast<__nv_bfloat16 *>(p.out)[oi] = __float2bfloat16_rn(v);
                else static_cast<float *>(p.out)[oi] = v;
            }
        }
        return;
    }

    if (p.cluster) {   // splits of this (row, group) form one cluster: combine on chip
#pragma unroll
        for (int o = 0; o < NO; ++o) {
            const int idx = tid + o * kAttnThreads;
            if (idx < G * HD) q_s[idx] = o_acc[o];
        }
        cluster_combine<HD>(p, true, q_s, m_s, l_s, r, g);
        return;
    }

    // partial (m, l, o) of this split
    constexpr int WS = HD + 4;
#pragma unroll
    for (int o = 0; o < NO; ++o) {
        const int idx = tid + o * kAttnThreads;
        if (idx < G * HD) {
            const int gi = idx / HD, d = idx - gi * HD;
            float *w = p.ws + (((size_t)r * p.n_q + hq0 + gi) * p.splits + sidx) * WS;
            w[4 + d] = o_acc[o];
            if (d == 0) {
                w[0] = m_s[gi];
                w[1] = l_s[gi];
            }
        }
    }
    __threadfence();
    __syncthreads();
    int *cnt = p.cnt + (size_t)r * p.n_kv + g;
    if (tid == 0) {
        const int old = atomicAdd(cnt, 1);
        flag_s = (old == nact - 1);
    }
    __syncthreads();
    if (!flag_s) return;
    __threadfence();
    for (int idx = tid; idx < G * HD; idx += kAttnThreads) {
        const int gi = idx / HD, d = idx - gi * HD;
        const float *w0 = p.ws + (((size_t)r * p.n_q + hq0 + gi) * p.splits) * WS;
        float M = -INFINITY;
        for (int c = 0; c < nact; ++c) M = fmaxf(M, __ldcg(w0 + (size_t)c * WS));
        float L = 0.f, O = 0.f;
        for (int c = 0; c < nact; ++c) {
            const float sc_c = expf(__ldcg(w0 + (size_t)c * WS) - M);
            L = fmaf(__ldcg(w0 + (size_t)c * WS + 1), sc_c, L);
            O = fmaf(__ldcg(w0 + (size_t)c * WS + 4 + d), sc_c, O);
        }
        const float v = O / L;
        const size_t oi = out_row + (size_t)(hq0 + gi) * HD + d;
        if (p.out_bf16) static_cast<__nv_bfloat16 *>(p.out)[oi] = __float2bfloat16_rn(v);
        else static_cast<float *>(p.out)[oi] = v;
    }
    if (tid == 0) *cnt = 0;
}

template <typename KT, int HD>
static cudaError_t launch_attn_t(const AttnParams &p, int rows, cudaStream_t st, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.splits, p.n_kv, rows);
    cfg.blockDim = dim3(kAttnThreads, 1, 1);
    cfg.dynamicSmemBytes = attn_smem_bytes(std::is_same<KT, int8_t>::value ? 2 : (sizeof(KT) == 2 ? 1 : 0), HD, p.group);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.cluster) {   // all splits of a (row, KV group) in one cluster
        if (p.splits > kAttnClusterMax) return cudaErrorInvalidValue;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = p.splits;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, k_attn_decode<KT, HD>, p);
}

cudaError_t launch_attn(int kv_kind, int head_dim, const AttnParams &p, int rows, cudaStream_t st, bool pdl) {
    if (attn_dec_keys_supported(kv_kind, head_dim, p)) return launch_attn_dec_keys(kv_kind, head_dim, p, rows, st, pdl);
    if (kv_kind == 2) {   // Q8_0 storage
        switch (head_dim) {
            case 64: return launch_attn_t<int8_t, 64>(p, rows, st, pdl);
            case 128: return launch_attn_t<int8_t, 128>(p, rows, st, pdl);
        }
        return cudaErrorInvalidValue;
    }
    if (kv_kind == 1) {
        switch (head_dim) {
            case 32: return launch_attn_t<__nv_bfloat16, 32>(p, rows, st, pdl);
            case 64: return launch_attn_t<__nv_bfloat16, 64>(p, rows, st, pdl);
            case 128: return launch_attn_t<__nv_bfloat16, 128>(p, rows, st, pdl);
        }
    } else {
        switch (head_dim) {
            case 32: return launch_attn_t<float, 32>(p, rows, st, pdl);
            case 64: return launch_attn_t<float, 64>(p, rows, st, pdl);
            case 128: return launch_attn_t<float, 128>(p, rows, st, pdl);
        }
    }
    return cudaErrorInvalidValue;
}

cudaError_t prepare_attn() {
    const int bytes = 200 * 1024;
    cudaError_t e = cudaSuccess;
    e = e ? e : cudaFuncSetAttribute(k_attn_decode<float, 32>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    e = e ? e : cudaFuncSetAttribute(k_attn_decode<float, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    e = e ? e : cudaFuncSetAttribute(k_attn_decode<float, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    e = e ? e : cudaFuncSetAttribute(k_attn_decode<__nv_bfloat16, 32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     bytes);
    e = e ? e : cudaFuncSetAttribute(k_attn_decode<__nv_bfloat16, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     bytes);
    e = e ? e : cudaFuncSetAttribute(k_attn_decode<__nv_bfloat16, 128>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    e = e ? e : cudaFuncSetAttribute(k_attn_decode<int8_t, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    e = e ? e : cudaFuncSetAttribute(k_attn_decode<int8_t, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    return e ? e : prepare_attn_dec_keys();
}

}  // namespace talker_k
