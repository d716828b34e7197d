// Decode attention over the paged bf16 KV cache, key-parallel form.
//
// For each decode row r (stream r at position p = cur_len[r]) and q head h of KV group g,
//   o_h = softmax_j(q_h . k_{g,j} / sqrt(hd)) v_{g,j},  j in [0, p]
// ("qwentts.cpp/src/talker-forward.h", talker_layer_forward: flash_attn_ext with F32
// precision over the causal window; GQA with G = n_q / n_kv q heads per KV head). The row's
// own k, v are appended at p first (set_rows); the window is bounded by p + 1, so cache rows
// past it never enter the arithmetic.
//
// Grid (splits, n_kv, rows), 8 warps. CTA (split, g, r) walks a contiguous range of 64-key
// pages of (stream r, layer, g); each page's K and V tiles are bulk-copied (TMA) into one of
// two slots, the copies of the first slots issued before the dependency wait. Warp w owns
// keys 8w .. 8w + 7 of every page and keeps its own online-softmax state (running maximum,
// sum and output in f32, base 2 with log2(e) folded into q):
//   scores: lane = (key, quarter of the head dimension); q for its quarter lives in registers;
//           the four quarters are summed with two shuffles;
//   P.V:    lane = HD/32 output dimensions; the warp's 8 probabilities come by shuffle.
// With bf16 storage and head_dim 128 the tiles come through the pool's tensor maps instead
// (128-byte swizzle, conflict-free 8 x 8 fragment loads) and a warp's 8 keys of a page go
// through the tensor cores (mma.sync; the M = 16 operand rows carry the G query heads twice):
//   scores: S[16 x 8 keys] = [hi(q); lo(q)] . K^T, m16n8k16 over the head dimension, with
//           q split into two bf16 parts (hi + lo) whose products sum to the f32 score;
//   P.V:    O[16 x 128] += [hi(p); lo(p)] . V, m16n8k8 over the warp's keys, V fragments by
//           transposing 8 x 8 loads; the two row halves add up to the f32 product.
// No CTA barrier separates the phases of a page; the warps meet only before a slot is
// refilled and once at the end, where their partials are merged. Splits combine either
// inside one thread-block cluster (every other rank pushes its partial into rank 0's shared
// memory and arrives on rank 0's mbarrier) or through L2 by the CTA that finishes last, with
// the same formula in both.
#include <math.h>

#include "common.cuh"
#include "kernels.cuh"
#include "tcgen05.cuh"

using namespace talker_dev;

namespace talker_k {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kSlotsBf16 = 2;                // page slots (K + V tiles) per CTA: bf16 tiles
constexpr int kSlotsQ8 = 4;                  // Q8_0 tiles (about half the bytes)
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t rank_addr(const void *local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    return remote;
}
__device__ __forceinline__ void st_rank_f32(uint32_t remote, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}
// Arrive on an mbarrier in another CTA of the cluster, releasing this CTA's earlier writes
// (made visible to the whole CTA by a preceding barrier) at cluster scope.
__device__ __forceinline__ void arrive_rank(uint32_t remote_bar) {
    asm volatile("fence.acq_rel.cluster;" ::: "memory");
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar) : "memory");
}

// Sub-chunk (16 bytes = 8 dims) that a lane reads in step i of its quarter, rotated so that
// the 8 lanes of one shared-memory phase (two keys x four quarters) hit distinct banks.
template <int HD>
__device__ __forceinline__ int rot(int i, int key, int quarter) {
    if constexpr (HD == 128) return (i + (quarter >> 1) + 2 * (key & 1)) & 3;
    else return (i + (key & 1)) & 1;
}

// Rotation of the two 16-byte halves of a lane's 32 Q8_0 codes (head_dim 128): the 8 lanes of a
// phase (two keys x four quarters) then hit distinct banks.
template <int HD>
__device__ __forceinline__ int rot_q8(int i, int key) {
    if constexpr (HD == 128) return (i + (key & 1)) & 1;
    else return i;
}

// The four signed codes of a 32-bit word as floats: each biased byte goes under the exponent
// of 2^23 (byte_perm), and subtracting 2^23 + 128 leaves the code exactly.
__device__ __forceinline__ void q8x4(uint32_t w, float *f) {
    const uint32_t v = w ^ 0x80808080u;
    f[0] = __int_as_float(__byte_perm(v, 0x4B000000u, 0x7440)) - 8388736.0f;
    f[1] = __int_as_float(__byte_perm(v, 0x4B000000u, 0x7441)) - 8388736.0f;
    f[2] = __int_as_float(__byte_perm(v, 0x4B000000u, 0x7442)) - 8388736.0f;
    f[3] = __int_as_float(__byte_perm(v, 0x4B000000u, 0x7443)) - 8388736.0f;
}

// Byte offset of (row, dim) in a bf16 [64][128] tile loaded as two 64-dim boxes with the
// 128-byte swizzle (16-byte chunk index XOR row % 8).
__device__ __forceinline__ uint32_t sw128(int row, int dim) {
    return (uint32_t)((dim >> 6) * 8192 + row * 128 + ((((dim & 63) >> 3) ^ (row & 7)) << 4) + (dim & 7) * 2);
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}
__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_1688(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
    asm("mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(b0));
}
// (lo, hi) as a bf16 pair, the first element in the low half
__device__ __forceinline__ uint32_t pack_bf16(__nv_bfloat16 lo, __nv_bfloat16 hi) {
    return (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
}
// x = hi + lo with both parts bf16 (hi the rounded value, lo the rounded remainder)
__device__ __forceinline__ void split_bf16(float x, __nv_bfloat16 &hi, __nv_bfloat16 &lo) {
    hi = __float2bfloat16_rn(x);
    lo = __float2bfloat16_rn(x - __bfloat162float(hi));
}

template <int G>
__device__ __forceinline__ void dot8(const uint4 u, const float (&q)[G][8], float (&s)[G]) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float t = s[g];
        t = fmaf(bf16lo(u.x), q[g][0], t);
        t = fmaf(bf16hi(u.x), q[g][1], t);
        t = fmaf(bf16lo(u.y), q[g][2], t);
        t = fmaf(bf16hi(u.y), q[g][3], t);
        t = fmaf(bf16lo(u.z), q[g][4], t);
        t = fmaf(bf16hi(u.z), q[g][5], t);
        t = fmaf(bf16lo(u.w), q[g][6], t);
        t = fmaf(bf16hi(u.w), q[g][7], t);
        s[g] = t;
    }
}

}  // namespace

// bf16 tile: [64][hd] values; Q8_0 tile: [64][hd] codes, then [64][hd / 32] fp16 scales.
// The tensor-core form (mm) aligns its swizzled tiles to 1024 bytes.
size_t attn_dec_keys_smem_bytes(int head_dim, int group, bool q8, bool mm) {
    const size_t tile = q8 ? (size_t)kPage * head_dim + (size_t)kPage * (head_dim / 32) * 2 : (size_t)kPage * head_dim * 2;
    const size_t gh = (size_t)group * head_dim;
    return 2 * (q8 ? kSlotsQ8 : kSlotsBf16) * tile + gh * 4 + 2 * (size_t)head_dim * 4 + kWarps * gh * 4 +
           kAttnClusterMax * (gh + 2 * group) * 4 + (mm ? 1024 : 0);
}

template <int HD, int G, bool Q8, bool MM>
__global__ void __launch_bounds__(kThreads, 2) k_attn_dec_keys(const AttnParams p, const __grid_constant__ KvMaps maps) {
    static_assert(!MM || (!Q8 && HD == 128 && G <= 8), "tensor-core form: bf16 tiles, head_dim 128, G <= 8");
    constexpr int QD = HD / 4;                 // dims of a key that one lane scores
    constexpr int EPL = Q8 ? 16 : 8;           // elements per 16-byte load
    constexpr int NSUB = QD / EPL;             // 16-byte loads per lane per key
    constexpr int PD = HD / 32;                // output dims per lane in P.V
    constexpr uint32_t kTile = Q8 ? kPage * HD + kPage * (HD / 32) * 2 : kPage * HD * 2;
    constexpr int kSlots = Q8 ? kSlotsQ8 : kSlotsBf16;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *kbuf = MM ? reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                                 ~(uintptr_t)1023)
                             : smem_raw;                              // [kSlots][tile]
    unsigned char *vbuf = kbuf + kSlots * kTile;                      // [kSlots][tile]
    float *q_s = reinterpret_cast<float *>(vbuf + kSlots * kTile);    // [G][HD], scaled
    float *knew = q_s + G * HD;                                       // this step's k, v row as stored
    float *vnew = knew + HD;
    float *ow = vnew + HD;                                            // [kWarps][G][HD] warp partials
    float *recv = ow + kWarps * G * HD;                               // [cluster rank][G*HD + 2G]
    constexpr int RS = G * HD + 2 * G;                                // floats per rank in recv
    __shared__ float wm[kWarps][G], wl[kWarps][G];
    __shared__ __align__(8) uint64_t bars[kSlots];
    __shared__ __align__(8) uint64_t cbar;                            // cluster rank 0: partials received
    __shared__ int flag_s;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int sidx = blockIdx.x, g = blockIdx.y, r = blockIdx.z;
    pdl_launch_dependents();
    // Before the wait only data of earlier launches is read: the length, the page table, the
    // RoPE table and the cached pages (the fresh row is patched in after the wait).
    const int pos = p.rowmap.cur_len[r];
    if (pos < 0 || pos >= p.cache.max_seq) {
        if (tid == 0 && sidx == 0) atomicOr(p.status, ST_BAD_POSITION);
        return;
    }
    const int nvis = pos + 1;
    const int npages = (nvis + kPage - 1) / kPage;
    const int per = (npages + p.splits - 1) / p.splits;
    const int pb = sidx * per;
    const int pe = min(pb + per, npages);
    const int nact = (npages + per - 1) / per;   // splits that hold pages
    const bool has = pb < pe;
    const bool clustered = p.cluster && nact > 1;
    if (!has && !clustered) return;

    const int *ptab = p.cache.page_table + (size_t)r * p.cache.pages_per_stream;
    // a (page, layer, head) tile is kTile contiguous bytes; page_elems counts pool units (bf16
    // elements, or bytes for Q8_0)
    const size_t head_off = (size_t)(p.layer * p.cache.n_kv + g) * kTile;
    const size_t page_bytes = p.cache.page_elems * (Q8 ? 1 : 2);
    unsigned char *kpool = static_cast<unsigned char *>(p.cache.k);
    unsigned char *vpool = static_cast<unsigned char *>(p.cache.v);
    auto tile_of = [&](unsigned char *pool, int page) { return pool + (size_t)page * page_bytes + head_off; };
    // tensor-map row of the tile's first key (tiles of all layers and heads of a page are consecutive)
    const int rows_per_page = (int)(p.cache.page_elems / HD);
    const int tile_row = (p.layer * p.cache.n_kv + g) * kPage;
    auto issue = [&](int slot, int page) {
        mbar_arrive_expect_tx(&bars[slot], 2 * kTile);
        if constexpr (MM) {
            const int y = page * rows_per_page + tile_row;
            tc::tma_load_2d(kbuf + slot * kTile, &maps.k, 0, y, &bars[slot]);
            tc::tma_load_2d(kbuf + slot * kTile + kTile / 2, &maps.k, 64, y, &bars[slot]);
            tc::tma_load_2d(vbuf + slot * kTile, &maps.v, 0, y, &bars[slot]);
            tc::tma_load_2d(vbuf + slot * kTile + kTile / 2, &maps.v, 64, y, &bars[slot]);
        } else {
            bulk_g2s(kbuf + slot * kTile, tile_of(kpool, page), kTile, &bars[slot]);
            bulk_g2s(vbuf + slot * kTile, tile_of(vpool, page), kTile, &bars[slot]);
        }
    };

    uint32_t rank = 0;
    if (clustered) asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
    if (tid == 0) {
        for (int b = 0; b < kSlots; ++b) mbar_init(&bars[b], 1);
        if (clustered && rank == 0) mbar_init(&cbar, nact - 1);   // one arrival per other active rank
        fence_barrier_init();
    }
    __syncthreads();
    if (tid == 0 && has) {
        for (int b = 0; b < kSlots && pb + b < pe; ++b) issue(b, ptab[pb + b]);
    }
    if (clustered) {
        // rank 0's receive barrier is initialised before any rank can arrive on it; ranks without
        // pages have nothing to send and leave here
        cluster_barrier();
        if (!has) return;
    }
    constexpr int half = HD / 2;
    float2 cs_pre[2] = {make_float2(1.f, 0.f), make_float2(1.f, 0.f)};
    if (warp <= G) {
#pragma unroll
        for (int j = 0; j < 2; ++j)
            if (lane + 32 * j < half) cs_pre[j] = p.rope[(size_t)pos * half + lane + 32 * j];
    }
    pdl_wait();

    // Heads of this group from the raw projections: q heads g*G.., k head g, v head g; QK-norm
    // and RoPE ("talker-forward.h", talker_layer_forward); split 0 appends k and v to the cache.
    const float qscale = p.scale * kLog2e;
    if (warp < G + 2) {
        const int hh = warp;
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
                    a[j] = x0 * cs_pre[j].x - x1 * cs_pre[j].y;
                    b[j] = x1 * cs_pre[j].x + x0 * cs_pre[j].y;
                }
            }
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int i = lane + 32 * j;
            if (i >= half) continue;
            if (hh < G) {
                q_s[hh * HD + i] = a[j] * qscale;
                q_s[hh * HD + i + half] = b[j] * qscale;
            } else {
                // the row as this step attends it: exact with Q8_0 storage (a call attends its own
                // rows unquantized), else as stored
                float *d = hh == G ? knew : vnew;
                d[i] = Q8 ? a[j] : Elem<__nv_bfloat16>::round(a[j]);
                d[i + half] = Q8 ? b[j] : Elem<__nv_bfloat16>::round(b[j]);
                if (!Q8 && sidx == 0) {
                    __nv_bfloat16 *c = reinterpret_cast<__nv_bfloat16 *>(tile_of(hh == G ? kpool : vpool, ptab[pos / kPage])) +
                                       (size_t)(pos % kPage) * HD;
                    c[i] = __float2bfloat16_rn(a[j]);
                    c[i + half] = __float2bfloat16_rn(b[j]);
                }
            }
        }
        if (Q8 && hh >= G && sidx == 0) {
            // Q8_0 row for later steps: each valid register of the warp is one block of 32 dims
            unsigned char *t = tile_of(hh == G ? kpool : vpool, ptab[pos / kPage]);
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
    __syncthreads();

    if constexpr (MM) {
        // Lane (h = lane / 4, c = 2 (lane % 4)): S rows h (hi) and h + 8 (lo) of keys c, c + 1 of
        // the warp's 8; the same lane holds O rows h, h + 8 of dims 8 n + c, c + 1 (n = 0..15).
        const int h = lane >> 2, c2 = (lane & 3) * 2;
        float mh = -INFINITY, lh = 0.f;
        float o[16][4];
#pragma unroll
        for (int n = 0; n < 16; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[n][e] = 0.f;
        bool failed = false;
        int fail_it = 0;
        if (has) {
            uint32_t qf[8][4];   // A fragments of [hi(q); lo(q)] per 16-dim step
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int d = ks * 16 + hf * 8 + c2;
                    const float x0 = h < G ? q_s[h * HD + d] : 0.f, x1 = h < G ? q_s[h * HD + d + 1] : 0.f;
                    __nv_bfloat16 h0, l0, h1, l1;
                    split_bf16(x0, h0, l0);
                    split_bf16(x1, h1, l1);
                    qf[ks][2 * hf] = pack_bf16(h0, h1);
                    qf[ks][2 * hf + 1] = pack_bf16(l0, l1);
                }
            const int lrow = warp * 8 + (lane & 7);   // the key row this lane addresses in 8 x 8 loads
            const int key0 = warp * 8 + c2;
            for (int pg = pb, it = 0; pg < pe; ++pg, ++it) {
                const int slot = it % kSlots;
                const bool ok = mbar_wait(&bars[slot], (it / kSlots) & 1, p.status);
                if (__syncthreads_or(!ok)) {
                    failed = true;
                    fail_it = it;
                    break;
                }
                unsigned char *Ks = kbuf + slot * kTile;
                unsigned char *Vs = vbuf + slot * kTile;
                const int valid = min(kPage, nvis - pg * kPage);
                const int newest = pos - pg * kPage;
                if (newest >= 0 && newest < kPage && (newest >> 3) == warp) {
                    // only this warp reads that row: patch the stored values in (the copy may predate them)
                    for (int i = lane; i < HD; i += 32) {
                        *reinterpret_cast<__nv_bfloat16 *>(Ks + sw128(newest, i)) = __float2bfloat16_rn(knew[i]);
                        *reinterpret_cast<__nv_bfloat16 *>(Vs + sw128(newest, i)) = __float2bfloat16_rn(vnew[i]);
                    }
                    __syncwarp();
                }
                const uint32_t kb = smem_u32(Ks), vb = smem_u32(Vs);
                float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int kp = 0; kp < 4; ++kp) {   // 32 dims: two m16n8k16 steps
                    uint32_t b[4];
                    ldsm_x4(kb + sw128(lrow, kp * 32 + (lane >> 3) * 8), b);
                    mma_16816(sc, qf[2 * kp], b[0], b[1]);
                    mma_16816(sc, qf[2 * kp + 1], b[2], b[3]);
                }
                const bool v0 = h < G && key0 < valid, v1 = h < G && key0 + 1 < valid;
                const float s0 = v0 ? sc[0] + sc[2] : -INFINITY, s1 = v1 ? sc[1] + sc[3] : -INFINITY;
                float mx = fmaxf(s0, s1);
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float m_new = fmaxf(mh, mx);
                const float alpha = (m_new == -INFINITY) ? 1.f : exp2f(mh - m_new);
                const float p0 = v0 ? exp2f(s0 - m_new) : 0.f, p1 = v1 ? exp2f(s1 - m_new) : 0.f;
                float ls = p0 + p1;
                ls += __shfl_xor_sync(0xffffffffu, ls, 1);
                ls += __shfl_xor_sync(0xffffffffu, ls, 2);
                lh = lh * alpha + ls;
                mh = m_new;
#pragma unroll
                for (int n = 0; n < 16; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) o[n][e] *= alpha;
                __nv_bfloat16 ph0, pl0, ph1, pl1;
                split_bf16(p0, ph0, pl0);
                split_bf16(p1, ph1, pl1);
                const uint32_t pa0 = pack_bf16(ph0, ph1), pa1 = pack_bf16(pl0, pl1);
                // keys past the window: their V values are never multiplied in (zeroed fragments)
                const bool partial = valid < kPage;
                const bool kv0 = key0 < valid, kv1 = key0 + 1 < valid;
                const uint32_t vmask = (kv0 ? 0x0000ffffu : 0u) | (kv1 ? 0xffff0000u : 0u);
#pragma unroll
                for (int j = 0; j < 4; ++j) {   // 32 dims: four m16n8k8 steps
                    uint32_t b[4];
                    ldsm_x4_t(vb + sw128(lrow, (4 * j + (lane >> 3)) * 8), b);
#pragma unroll
                    for (int u = 0; u < 4; ++u) mma_1688(o[4 * j + u], pa0, pa1, partial ? b[u] & vmask : b[u]);
                }
                if (pg + kSlots < pe) {   // refill this slot once every warp is done with it
                    __syncthreads();
                    if (tid == 0) {
                        fence_proxy_async();
                        issue(slot, ptab[pg + kSlots]);
                    }
                }
            }
            if (failed) {
                if (tid == 0)
                    for (int j = fail_it; j < fail_it + kSlots && pb + j < pe; ++j)
                        mbar_wait(&bars[j % kSlots], (j / kSlots) & 1, p.status);
                __syncthreads();
                mh = -INFINITY;
                lh = 0.f;
#pragma unroll
                for (int n = 0; n < 16; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) o[n][e] = 0.f;
            }
        }
        // this warp's partial: lane 4h holds (m, l) of head h, rows h and h + 8 sum to O
        if (h < G) {
            if ((lane & 3) == 0) {
                wm[warp][h] = mh;
                wl[warp][h] = lh;
            }
#pragma unroll
            for (int n = 0; n < 16; ++n) {
                float *dst = ow + (warp * G + h) * HD + n * 8 + c2;
                dst[0] = o[n][0] + o[n][2];
                dst[1] = o[n][1] + o[n][3];
            }
        }
    } else {
        // per-warp online softmax state
        float m[G], l[G], o[G][PD];
    #pragma unroll
        for (int gi = 0; gi < G; ++gi) {
            m[gi] = -INFINITY;
            l[gi] = 0.f;
    #pragma unroll
            for (int d = 0; d < PD; ++d) o[gi][d] = 0.f;
        }
        const int kk = warp * 8 + (lane >> 2), quarter = lane & 3;
        bool failed = false;
        int fail_it = 0;
        if (has) {
            float qr[G][NSUB][EPL];   // q over this lane's quarter, in the lane's load order
            auto sub_of = [&](int i) { return Q8 ? rot_q8<HD>(i, kk) : rot<HD>(i, kk, quarter); };
    #pragma unroll
            for (int gi = 0; gi < G; ++gi)
    #pragma unroll
                for (int i = 0; i < NSUB; ++i) {
                    const float *qs = q_s + gi * HD + quarter * QD + sub_of(i) * EPL;
    #pragma unroll
                    for (int e = 0; e < EPL; ++e) qr[gi][i][e] = qs[e];
                }
            for (int pg = pb, it = 0; pg < pe; ++pg, ++it) {
                const int slot = it % kSlots;
                const bool ok = mbar_wait(&bars[slot], (it / kSlots) & 1, p.status);
                if (__syncthreads_or(!ok)) {
                    failed = true;
                    fail_it = it;
                    break;
                }
                unsigned char *Ks = kbuf + slot * kTile;
                unsigned char *Vs = vbuf + slot * kTile;
                const int valid = min(kPage, nvis - pg * kPage);
                const int newest = pos - pg * kPage;   // the fresh row, when this page holds it
                if (!Q8 && newest >= 0 && newest < kPage && (newest >> 3) == warp) {
                    // only this warp reads that row: patch the stored values in (the copy may predate them)
                    __nv_bfloat16 *kr = reinterpret_cast<__nv_bfloat16 *>(Ks) + newest * HD;
                    __nv_bfloat16 *vr = reinterpret_cast<__nv_bfloat16 *>(Vs) + newest * HD;
                    for (int i = lane; i < HD; i += 32) {
                        kr[i] = __float2bfloat16_rn(knew[i]);
                        vr[i] = __float2bfloat16_rn(vnew[i]);
                    }
                    __syncwarp();
                }
                // scores of key kk for every head
                float sc[G];
    #pragma unroll
                for (int gi = 0; gi < G; ++gi) sc[gi] = 0.f;
                if constexpr (!Q8) {
                    const uint32_t krow = smem_u32(Ks) + (uint32_t)(kk * HD + quarter * QD) * 2;
    #pragma unroll
                    for (int i = 0; i < NSUB; ++i) {
                        const uint4 u = lds_u4(krow + rot<HD>(i, kk, quarter) * 16);
                        float qv[G][8];
    #pragma unroll
                        for (int gi = 0; gi < G; ++gi)
    #pragma unroll
                            for (int e = 0; e < 8; ++e) qv[gi][e] = qr[gi][i][e];
                        dot8<G>(u, qv, sc);
                    }
                } else if (kk == newest) {   // this step's own row, exact
    #pragma unroll
                    for (int i = 0; i < NSUB; ++i)
    #pragma unroll
                        for (int e = 0; e < EPL; ++e) {
                            const float x = knew[quarter * QD + sub_of(i) * EPL + e];
    #pragma unroll
                            for (int gi = 0; gi < G; ++gi) sc[gi] = fmaf(qr[gi][i][e], x, sc[gi]);
                        }
                } else {   // codes times q, then the block's scale
                    const uint32_t krow = smem_u32(Ks) + (uint32_t)(kk * HD + quarter * QD);
    #pragma unroll
                    for (int i = 0; i < NSUB; ++i) {
                        const uint4 u = lds_u4(krow + sub_of(i) * 16);
                        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
    #pragma unroll
                        for (int wq = 0; wq < 4; ++wq) {
                            float c4[4];
                            q8x4(w4[wq], c4);
    #pragma unroll
                            for (int e = 0; e < 4; ++e)
    #pragma unroll
                                for (int gi = 0; gi < G; ++gi) sc[gi] = fmaf(qr[gi][i][wq * 4 + e], c4[e], sc[gi]);
                        }
                    }
                    const float sd = __half2float(*reinterpret_cast<const __half *>(
                        Ks + kPage * HD + (kk * (HD / 32) + (quarter * QD) / 32) * 2));
    #pragma unroll
                    for (int gi = 0; gi < G; ++gi) sc[gi] *= sd;
                }
                const bool kval = kk < valid;
                float pk[G];
    #pragma unroll
                for (int gi = 0; gi < G; ++gi) {
                    float s = sc[gi];
                    s += __shfl_xor_sync(0xffffffffu, s, 1);
                    s += __shfl_xor_sync(0xffffffffu, s, 2);
                    s = kval ? s : -INFINITY;
                    float mx = s;
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                    const float m_new = fmaxf(m[gi], mx);
                    const float alpha = (m_new == -INFINITY) ? 1.f : exp2f(m[gi] - m_new);
                    pk[gi] = kval ? exp2f(s - m_new) : 0.f;
                    float ls = pk[gi];
                    ls += __shfl_xor_sync(0xffffffffu, ls, 4);
                    ls += __shfl_xor_sync(0xffffffffu, ls, 8);
                    ls += __shfl_xor_sync(0xffffffffu, ls, 16);
                    l[gi] = l[gi] * alpha + ls;
                    m[gi] = m_new;
    #pragma unroll
                    for (int d = 0; d < PD; ++d) o[gi][d] *= alpha;
                }
                // P.V over the warp's 8 keys (rows past the window are skipped: their contents are
                // never read into the arithmetic)
                const uint32_t vbase = smem_u32(Vs) + (uint32_t)(lane * PD) * (Q8 ? 1 : 2);
    #pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int key = warp * 8 + j;
                    float pj[G];
    #pragma unroll
                    for (int gi = 0; gi < G; ++gi) pj[gi] = __shfl_sync(0xffffffffu, pk[gi], j * 4);
                    if (key < valid) {
                        float v[PD];
                        if constexpr (Q8) {
                            if (key == newest) {   // this step's own row, exact
    #pragma unroll
                                for (int d = 0; d < PD; ++d) v[d] = vnew[lane * PD + d];
                            } else {
                                float c4[4];
                                uint32_t w;
                                if constexpr (PD == 4) asm("ld.shared.u32 %0, [%1];" : "=r"(w) : "r"(vbase + (uint32_t)key * HD));
                                else w = lds_u16(vbase + (uint32_t)key * HD);
                                q8x4(w, c4);
                                const float sd = __half2float(*reinterpret_cast<const __half *>(
                                    Vs + kPage * HD + (key * (HD / 32) + (lane * PD) / 32) * 2));
    #pragma unroll
                                for (int d = 0; d < PD; ++d) v[d] = c4[d] * sd;
                            }
                        } else if constexpr (PD == 4) {
                            const uint2 u = lds_u2(vbase + (uint32_t)key * HD * 2);
                            v[0] = bf16lo(u.x);
                            v[1] = bf16hi(u.x);
                            v[2] = bf16lo(u.y);
                            v[3] = bf16hi(u.y);
                        } else {
                            uint32_t u;
                            asm("ld.shared.u32 %0, [%1];" : "=r"(u) : "r"(vbase + (uint32_t)key * HD * 2));
                            v[0] = bf16lo(u);
                            v[1] = bf16hi(u);
                        }
    #pragma unroll
                        for (int gi = 0; gi < G; ++gi)
    #pragma unroll
                            for (int d = 0; d < PD; ++d) o[gi][d] = fmaf(pj[gi], v[d], o[gi][d]);
                    }
                }
                if (pg + kSlots < pe) {   // refill this slot once every warp is done with it
                    __syncthreads();
                    if (tid == 0) {
                        fence_proxy_async();
                        issue(slot, ptab[pg + kSlots]);
                    }
                }
            }
            if (failed) {
                // give the copies still in flight a bounded chance to land before the CTA moves on
                if (tid == 0)
                    for (int j = fail_it; j < fail_it + kSlots && pb + j < pe; ++j)
                        mbar_wait(&bars[j % kSlots], (j / kSlots) & 1, p.status);
                __syncthreads();
    #pragma unroll
                for (int gi = 0; gi < G; ++gi) {
                    m[gi] = -INFINITY;
                    l[gi] = 0.f;
    #pragma unroll
                    for (int d = 0; d < PD; ++d) o[gi][d] = 0.f;
                }
            }
        }

        // merge the warps (one barrier): thread t takes output t, scaling each warp's partial by
        // 2^(m_w - M) and adding them in warp order (deterministic)
        if (lane == 0) {
    #pragma unroll
            for (int gi = 0; gi < G; ++gi) {
                wm[warp][gi] = m[gi];
                wl[warp][gi] = l[gi];
            }
        }
    #pragma unroll
        for (int gi = 0; gi < G; ++gi)
    #pragma unroll
            for (int d = 0; d < PD; ++d) ow[(warp * G + gi) * HD + lane * PD + d] = o[gi][d];
    }
    __syncthreads();

    const int hq0 = g * G;
    const size_t out_row = (size_t)r * p.n_q * HD;
    auto store = [&](int idx, float v) {
        const int gi = idx / HD, d = idx - gi * HD;
        const size_t oi = out_row + (size_t)(hq0 + gi) * HD + d;
        if (p.out_bf16) static_cast<__nv_bfloat16 *>(p.out)[oi] = __float2bfloat16_rn(v);
        else static_cast<float *>(p.out)[oi] = v;
    };
    constexpr int kPer = (G * HD + kThreads - 1) / kThreads;   // outputs per thread
    float Mx[kPer], Lx[kPer], Ox[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const int idx = tid + u * kThreads;
        Mx[u] = -INFINITY;
        Lx[u] = 0.f;
        Ox[u] = 0.f;
        if (idx < G * HD) {
            const int gi = idx / HD;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) Mx[u] = fmaxf(Mx[u], wm[w][gi]);
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float e = (wm[w][gi] == -INFINITY) ? 0.f : exp2f(wm[w][gi] - Mx[u]);
                Lx[u] = fmaf(wl[w][gi], e, Lx[u]);
                Ox[u] = fmaf(ow[w * G * HD + idx], e, Ox[u]);
            }
        }
    }
    if (nact == 1) {
#pragma unroll
        for (int u = 0; u < kPer; ++u)
            if (tid + u * kThreads < G * HD) store(tid + u * kThreads, Ox[u] / Lx[u]);
        return;
    }
    if (clustered) {
        // ranks 1 .. nact-1 push their (M, L, O) into rank 0's receive area and arrive on its
        // barrier; rank 0 combines them with its own in rank order
        if (rank != 0) {
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
                const int idx = tid + u * kThreads;
                if (idx < G * HD) {
                    float *dst = recv + rank * RS;
                    st_rank_f32(rank_addr(dst + idx, 0), Ox[u]);
                    if (idx % HD == 0) {
                        st_rank_f32(rank_addr(dst + G * HD + idx / HD, 0), Mx[u]);
                        st_rank_f32(rank_addr(dst + G * HD + G + idx / HD, 0), Lx[u]);
                    }
                }
            }
            __syncthreads();
            if (tid == 0) arrive_rank(rank_addr(&cbar, 0));
            return;
        }
        const bool ok = mbar_wait(&cbar, 0, p.status);
        asm volatile("fence.acq_rel.cluster;" ::: "memory");   // the other ranks' pushes are visible
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int idx = tid + u * kThreads;
            if (idx >= G * HD || !ok) continue;
            const int gi = idx / HD;
            float M = Mx[u];
            for (int c = 1; c < nact; ++c) M = fmaxf(M, recv[c * RS + G * HD + gi]);
            float L = (Mx[u] == -INFINITY) ? 0.f : Lx[u] * exp2f(Mx[u] - M);
            float O = (Mx[u] == -INFINITY) ? 0.f : Ox[u] * exp2f(Mx[u] - M);
            for (int c = 1; c < nact; ++c) {
                const float mc = recv[c * RS + G * HD + gi];
                const float e = (mc == -INFINITY) ? 0.f : exp2f(mc - M);
                L = fmaf(recv[c * RS + G * HD + G + gi], e, L);
                O = fmaf(recv[c * RS + idx], e, O);
            }
            store(idx, O / L);
        }
        return;
    }
    // through L2: partial (M, L, O) of this split, the CTA that arrives last combines in split order
    constexpr int WS = HD + 4;
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const int idx = tid + u * kThreads;
        if (idx < G * HD) {
            const int gi = idx / HD, d = idx - gi * HD;
            float *wsp = p.ws + (((size_t)r * p.n_q + hq0 + gi) * p.splits + sidx) * WS;
            wsp[4 + d] = Ox[u];
            if (d == 0) {
                wsp[0] = Mx[u];
                wsp[1] = Lx[u];
            }
        }
    }
    __threadfence();
    __syncthreads();
    int *cnt = p.cnt + (size_t)r * p.n_kv + g;
    if (tid == 0) flag_s = (atomicAdd(cnt, 1) == nact - 1);
    __syncthreads();
    if (!flag_s) return;
    __threadfence();
    // Eight splits' partials are requested at a time (independent loads in flight), so the
    // combine costs a few L2 round trips, not one per split.
    constexpr int CB = 8;
    for (int idx = tid; idx < G * HD; idx += kThreads) {
        const int gi = idx / HD, d = idx - gi * HD;
        const float *w0 = p.ws + (((size_t)r * p.n_q + hq0 + gi) * p.splits) * WS;
        float M = -INFINITY;
        for (int c0 = 0; c0 < nact; c0 += CB) {
            float mv[CB];
#pragma unroll
            for (int c = 0; c < CB; ++c) mv[c] = c0 + c < nact ? __ldcg(w0 + (size_t)(c0 + c) * WS) : -INFINITY;
#pragma unroll
            for (int c = 0; c < CB; ++c) M = fmaxf(M, mv[c]);
        }
        float L = 0.f, O = 0.f;
        for (int c0 = 0; c0 < nact; c0 += CB) {
            float mv[CB], lv[CB], ov[CB];
#pragma unroll
            for (int c = 0; c < CB; ++c) {
                const bool in = c0 + c < nact;
                const float *wc = w0 + (size_t)(c0 + c) * WS;
                mv[c] = in ? __ldcg(wc) : -INFINITY;
                lv[c] = in ? __ldcg(wc + 1) : 0.f;
                ov[c] = in ? __ldcg(wc + 4 + d) : 0.f;
            }
#pragma unroll
            for (int c = 0; c < CB; ++c) {
                const float e = (mv[c] == -INFINITY) ? 0.f : exp2f(mv[c] - M);
                L = fmaf(lv[c], e, L);
                O = fmaf(ov[c], e, O);
            }
        }
        store(idx, O / L);
    }
    if (tid == 0) *cnt = 0;
}

bool attn_dec_keys_supported(int kv_kind, int head_dim, const AttnParams &p) {
    return (kv_kind == 1 || kv_kind == 2) && (head_dim == 64 || head_dim == 128) && (p.group == 1 || p.group == 2) &&
           p.rowmap.mode == 0 && p.raw != nullptr && (!p.cluster || p.splits <= kAttnClusterMax);
}

template <int HD, int G, bool Q8, bool MM>
static cudaError_t launch_keys_t(const AttnParams &p, int rows, cudaStream_t st, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.splits, p.n_kv, rows);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = attn_dec_keys_smem_bytes(HD, G, Q8, MM);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.cluster) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = p.splits;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    static const KvMaps none{};
    return cudaLaunchKernelEx(&cfg, k_attn_dec_keys<HD, G, Q8, MM>, p, MM ? *p.cache.maps : none);
}

template <bool Q8>
static cudaError_t launch_keys_q(int head_dim, const AttnParams &p, int rows, cudaStream_t st, bool pdl) {
    if (head_dim == 128) {
        if (!Q8 && p.cache.maps != nullptr)   // bf16 tiles through the tensor maps, tensor-core scores and P.V
            return p.group == 2 ? launch_keys_t<128, 2, false, true>(p, rows, st, pdl)
                                : launch_keys_t<128, 1, false, true>(p, rows, st, pdl);
        return p.group == 2 ? launch_keys_t<128, 2, Q8, false>(p, rows, st, pdl)
                            : launch_keys_t<128, 1, Q8, false>(p, rows, st, pdl);
    }
    if (head_dim == 64)
        return p.group == 2 ? launch_keys_t<64, 2, Q8, false>(p, rows, st, pdl)
                            : launch_keys_t<64, 1, Q8, false>(p, rows, st, pdl);
    return cudaErrorInvalidValue;
}

cudaError_t launch_attn_dec_keys(int kv_kind, int head_dim, const AttnParams &p, int rows, cudaStream_t st, bool pdl) {
    return kv_kind == 2 ? launch_keys_q<true>(head_dim, p, rows, st, pdl) : launch_keys_q<false>(head_dim, p, rows, st, pdl);
}

template <int HD, int G, bool Q8, bool MM>
static cudaError_t raise_one() {
    return cudaFuncSetAttribute(k_attn_dec_keys<HD, G, Q8, MM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)attn_dec_keys_smem_bytes(HD, G, Q8, MM));
}

cudaError_t prepare_attn_dec_keys() {
    cudaError_t e = raise_one<128, 2, false, false>();
    e = e ? e : raise_one<128, 1, false, false>();
    e = e ? e : raise_one<64, 2, false, false>();
    e = e ? e : raise_one<64, 1, false, false>();
    e = e ? e : raise_one<128, 2, true, false>();
    e = e ? e : raise_one<128, 1, true, false>();
    e = e ? e : raise_one<64, 2, true, false>();
    e = e ? e : raise_one<64, 1, true, false>();
    e = e ? e : raise_one<128, 2, false, true>();
    return e ? e : raise_one<128, 1, false, true>();
}

}  // namespace talker_k
