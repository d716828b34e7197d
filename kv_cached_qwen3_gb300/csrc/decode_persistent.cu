// Persistent decode kernel: one whole decode step (all layers + head) in one
// cooperative launch with one CTA per SM.
//
// Math per layer ("qwentts.cpp/src/talker-forward.h", talker_layer_forward and
// talker_layer_forward_batch, one row per stream at position cur_len[s]):
//   h = rmsnorm(x) * w_in;  [q;k;v] = W_qkv h;  q,k <- per-head rmsnorm * gain, NEOX RoPE;
//   k,v -> cache row cur_len;  o = softmax(q K^T / sqrt(hd)) V over [0, cur_len];
//   x += W_o o;  h2 = rmsnorm(x) * w_post;  x += W_d (silu(W_g h2) * (W_u h2))
// then y = rmsnorm(x) * w_final, logits = W_c y, argmax, cur_len += 1.
//
// Structure. Warp 16 of each CTA is a producer: one lane walks the CTA's fixed
// schedule of weight chunks (its contiguous, balanced share of every weight
// matrix of every layer) and KV pages (its attention split), and moves each
// into a ring of shared-memory slots with bulk (TMA) copies. Weights and the
// already-cached KV rows do not depend on this step's activations, so the
// stream of HBM reads never waits on the phases. Warps 0..15 are consumers:
// they run the phases QKV -> attention -> o_proj -> gate/up -> down per layer,
// reading the activations they need from L2 after a grid barrier, and free
// ring slots as they go. The attention phase waits only for the rows of its
// own KV group (per-head row counters), not for a full barrier.
//
// Every wait is bounded (1 s). A wait that gives up sets the device status
// word and a global abort flag; from then on every wait of every CTA returns
// at once, the control flow of all threads stays the same, and the kernel runs
// to its end (its outputs are then meaningless and the status says so).
#include <math.h>

#include "common.cuh"
#include "kernels.cuh"

using namespace talker_dev;

namespace talker_k {
namespace pk {

constexpr int NCW = 15;             // consumer warps
constexpr int NCT = NCW * 32;       // consumer threads
constexpr int NT = NCT + 32;        // + one producer warp
constexpr int SLOT = 32 * 1024;     // ring slot bytes
constexpr int NS = 5;               // ring slots
constexpr int MAXG = 8;             // max q heads per KV group

// Sync words (ints) in PersistParams::sync.
enum : int { SY_BAR = 0, SY_EXIT = 1, SY_ABORT = 2, SY_HEAD = 3, SY_ROWS = 8 };

__device__ __forceinline__ void cbar() { asm volatile("bar.sync 1, %0;" ::"n"(NCT) : "memory"); }

__device__ __forceinline__ int ld_acquire(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ int ld_volatile(const int *p) {
    int v;
    asm volatile("ld.volatile.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_add(int *p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

struct Ctx {
    volatile int *abort_s;   // CTA-local sticky abort flag (shared memory)
    int *abort_g;            // global abort flag
    int *status;
};

__device__ __forceinline__ void raise_abort(const Ctx &c) {
    *c.abort_s = 1;
    atomicExch(c.abort_g, 1);
    atomicOr(c.status, ST_WAIT_TIMEOUT);
}

// mbarrier wait that degrades to a no-op once the CTA or the grid has aborted.
__device__ __forceinline__ void ring_wait(uint64_t *bar, uint32_t parity, const Ctx &c) {
    if (*c.abort_s) return;
    if (mbar_try_wait(bar, parity)) return;
    const long long t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return;
        if ((it & 255) == 0) {
            if (*c.abort_s || ld_volatile(c.abort_g)) {
                *c.abort_s = 1;
                return;
            }
            if (clock64() - t0 > kWaitLimitCycles) {
                raise_abort(c);
                return;
            }
        }
    }
}

// Single-thread spin until *ctr >= target (acquire), bounded and abort-aware.
__device__ __forceinline__ void spin_geq(const int *ctr, int target, const Ctx &c) {
    if (*c.abort_s) return;
    if (ld_acquire(ctr) >= target) return;
    const long long t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (ld_acquire(ctr) >= target) return;
        if ((it & 63) == 0) {
            if (ld_volatile(c.abort_g)) {
                *c.abort_s = 1;
                return;
            }
            if (clock64() - t0 > kWaitLimitCycles) {
                raise_abort(c);
                return;
            }
        }
    }
}

// Grid barrier among the consumer warps of all CTAs (arrival count is monotonic within a launch).
__device__ __forceinline__ void grid_barrier(int *bar, int target, const Ctx &c, int ctid) {
    cbar();
    if (ctid == 0) {
        __threadfence();
        red_release_add(bar, 1);
        spin_geq(bar, target, c);
        __threadfence();
    }
    cbar();
}

struct Span {
    int u0, n;
};
// Contiguous, balanced share of N units for CTA `cta` out of P.
__device__ __forceinline__ Span cta_span(int N, int cta, int P) {
    // 32-bit division only (a 64-bit division costs hundreds of cycles); N * P < 2^32 is
    // checked on the host
    const int a = (int)((unsigned)N * (unsigned)cta / (unsigned)P);
    const int b = (int)((unsigned)N * (unsigned)(cta + 1) / (unsigned)P);
    return {a, b - a};
}

using LayerW = PersistLayer;

}  // namespace pk
}  // namespace talker_k

namespace talker_k {
namespace pk {

// Attention work of one CTA: query row r (stream r), KV group g, split `split`
// of S over the pages [0, npages) of positions [0, pos].
struct AttnWork {
    int has, r, g, split, S, pos, pb, pe, nact;
};

__device__ __forceinline__ AttnWork attn_work(const PersistParams &p, int cta, int P, const int *curlen_s) {
    AttnWork w{};
    const int items = p.rows * p.nkv;
    const int S = p.splits;
    if (cta >= items * S) return w;
    const int item = cta % items;
    w.r = item / p.nkv;
    w.g = item % p.nkv;
    w.split = cta / items;
    w.S = S;
    w.pos = curlen_s[w.r];
    if (w.pos < 0 || w.pos >= p.cache.max_seq) return w;   // host checks make this unreachable
    const int npages = (w.pos + 1 + kPage - 1) / kPage;
    const int per = (npages + S - 1) / S;
    w.pb = w.split * per;
    w.pe = min(w.pb + per, npages);
    w.nact = (npages + per - 1) / per;
    w.has = w.pb < w.pe;
    return w;
}

// The producer lane: streams the CTA's schedule into the ring, in exactly the
// order the consumers read it.
template <typename WT, typename KT, int HD>
__device__ void producer(const PersistParams &p, unsigned char *ring, uint64_t *full, uint64_t *empty, const Ctx &c,
                         const AttnWork &aw) {
    const int P = gridDim.x, cta = blockIdx.x;
    const size_t wsz = sizeof(WT);
    const int qkv_n = (p.nq + 2 * p.nkv) * p.hd;
    unsigned long long *trace = p.trace != nullptr ? p.trace + (size_t)cta * kTraceSlots : nullptr;
    uint32_t k = 0;
    // With tracing on, the producer stamps when each issued chunk has landed (seen while it waits).
    uint32_t landed = 0;
    auto poll_landed = [&]() {
        while (landed < k && mbar_test_wait(&full[landed % NS], (landed / NS) & 1)) {
            if (landed < (uint32_t)kTraceChunks) trace[kTraceDots + landed] = clock64();
            ++landed;
        }
    };
    auto issue = [&](const void *s1, uint32_t b1, const void *s2, uint32_t b2) {
        const int slot = k % NS;
        const uint32_t use = k / NS;
        if (use > 0) {
            if (trace)
                for (int it = 0; it < (1 << 20) && !mbar_test_wait(&empty[slot], (use - 1) & 1); ++it) poll_landed();
            ring_wait(&empty[slot], (use - 1) & 1, c);
        }
        if (trace && k < (uint32_t)kTraceChunks) trace[kTraceProducer + k] = clock64();
        if (!*c.abort_s) {
            unsigned char *dst = ring + (size_t)slot * SLOT;
            mbar_arrive_expect_tx(&full[slot], b1 + b2);
            bulk_g2s(dst, s1, b1, &full[slot]);
            if (b2) bulk_g2s(dst + b1, s2, b2, &full[slot]);
        }
        ++k;
    };
    auto stream_rows = [&](const void *W, int N, size_t unit_bytes) {
        const Span s = cta_span(N, cta, P);
        const int upc = max(1, (int)(SLOT / unit_bytes));
        for (int u = s.u0; u < s.u0 + s.n; u += upc) {
            const int n = min(upc, s.u0 + s.n - u);
            issue(static_cast<const char *>(W) + (size_t)u * unit_bytes, (uint32_t)(n * unit_bytes), nullptr, 0);
        }
    };
    const uint32_t tile = kPage * HD * sizeof(KT);
    const KT *kpool = static_cast<const KT *>(p.cache.k);
    const KT *vpool = static_cast<const KT *>(p.cache.v);
    for (int l = 0; l < p.n_layers; ++l) {
        const LayerW &L = p.layers[l];
        stream_rows(L.qkv, qkv_n, (size_t)p.H * wsz);
        if (aw.has) {
            const int *ptab = p.cache.page_table + (size_t)aw.r * p.cache.pages_per_stream;
            const size_t head_off = (size_t)(l * p.cache.n_kv + aw.g) * kPage * HD;
            for (int pg = aw.pb; pg < aw.pe; ++pg) {
                const size_t off = (size_t)ptab[pg] * p.cache.page_elems + head_off;
                issue(kpool + off, tile, vpool + off, tile);
            }
        }
        stream_rows(L.o, p.H, (size_t)p.nq * p.hd * wsz);
        stream_rows(L.gu, p.I, (size_t)2 * p.H * wsz);
        stream_rows(L.down, p.H, (size_t)p.I * wsz);
    }
    stream_rows(p.head, p.V, (size_t)p.H * wsz);
    // Let the last copies land before the CTA may exit.
    for (uint32_t j = (k > (uint32_t)NS ? k - NS : 0); j < k; ++j) ring_wait(&full[j % NS], (j / NS) & 1, c);
}

// Consumer-side ring cursor.
struct Ring {
    unsigned char *base;
    uint64_t *full, *empty;
    uint32_t k;
    unsigned long long *trace;   // this CTA's trace row (consumer thread 0 only) or null
    __device__ __forceinline__ const unsigned char *acquire(const Ctx &c) {
        ring_wait(&full[k % NS], (k / NS) & 1, c);
        if (trace && k < (uint32_t)kTraceChunks) trace[kTraceAcquire + k] = clock64();
        return base + (size_t)(k % NS) * SLOT;
    }
    // Every consumer warp arrives once per slot (the empty barrier counts NCW arrivals).
    __device__ __forceinline__ void release(int lane) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[k % NS]);
        ++k;
    }
};

template <int EPV>
__device__ __forceinline__ int aidx(int r, int k, int K) {
    if (EPV == 8) return r * K + ((k >> 2) & 1) * (K >> 1) + (k >> 3) * 4 + (k & 3);
    return r * K + k;
}

// Stage rows x[0..rows) of width K (row stride ld) into `act` in the vector
// layout of the dot products; with `gain`, apply RMSNorm and the gain
// (x / sqrt(mean(x^2) + eps) * gain). Ends with a consumer barrier.
template <int EPV, int R>
__device__ void stage(float *act, const float *src, int ld, int K, int rows, const float *gain, float eps,
                      float *red, int ctid) {
    const int K4 = K >> 2;
    const int warp = ctid >> 5, lane = ctid & 31;
    float ss[R];
#pragma unroll
    for (int r = 0; r < R; ++r) ss[r] = 0.f;
    cbar();   // every warp is done reading the previous contents of act
    for (int idx = ctid; idx < rows * K4; idx += NCT) {
        const int r = idx / K4, k = (idx - r * K4) * 4;
        const float4 v = __ldcg(reinterpret_cast<const float4 *>(src + (size_t)r * ld + k));
        *reinterpret_cast<float4 *>(act + aidx<EPV>(r, k, K)) = v;
        const float s = v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
#pragma unroll
        for (int rr = 0; rr < R; ++rr)
            if (rr == r) ss[rr] += s;
    }
    if (gain != nullptr) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float v = warp_sum(ss[r]);
            if (lane == 0) red[warp * R + r] = v;
        }
        cbar();
        float inv[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float t = 0.f;
            for (int w = 0; w < NCW; ++w) t += red[w * R + r];
            inv[r] = 1.0f / sqrtf(t / (float)K + eps);
        }
        for (int idx = ctid; idx < rows * K4; idx += NCT) {
            const int r = idx / K4, k = (idx - r * K4) * 4;
            float4 *a = reinterpret_cast<float4 *>(act + aidx<EPV>(r, k, K));
            float4 v = *a;
            float iv = inv[0];
#pragma unroll
            for (int rr = 1; rr < R; ++rr)
                if (rr == r) iv = inv[rr];
            v.x = v.x * iv * gain[k];
            v.y = v.y * iv * gain[k + 1];
            v.z = v.z * iv * gain[k + 2];
            v.w = v.w * iv * gain[k + 3];
            *a = v;
        }
    }
    cbar();
}

// acc[n][r] = sum_k W[n][k] * act[r][k] for NU consecutive weight rows in shared memory.
template <typename WT, int R, int NU>
__device__ __forceinline__ void dot_rows(const unsigned char *w, int K, const float *act, int rows, float (&acc)[NU][R],
                                         int lane) {
    constexpr int EPV = Elem<WT>::kPerVec;
#pragma unroll
    for (int n = 0; n < NU; ++n)
#pragma unroll
        for (int r = 0; r < R; ++r) acc[n][r] = 0.f;
    const int nvec = K / EPV;
    const size_t row_bytes = (size_t)K * sizeof(WT);
    for (int v = lane; v < nvec; v += 32) {
        uint4 wv[NU];
#pragma unroll
        for (int n = 0; n < NU; ++n) wv[n] = *reinterpret_cast<const uint4 *>(w + n * row_bytes + (size_t)v * 16);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (r < rows) {
                if (EPV == 8) {
                    const float4 a0 = *reinterpret_cast<const float4 *>(act + r * K + v * 4);
                    const float4 a1 = *reinterpret_cast<const float4 *>(act + r * K + (K >> 1) + v * 4);
#pragma unroll
                    for (int n = 0; n < NU; ++n) {
                        const uint4 u = wv[n];
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
                    const float4 a0 = *reinterpret_cast<const float4 *>(act + r * K + v * 4);
#pragma unroll
                    for (int n = 0; n < NU; ++n) {
                        const uint4 u = wv[n];
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
#pragma unroll
    for (int n = 0; n < NU; ++n)
#pragma unroll
        for (int r = 0; r < R; ++r) acc[n][r] = warp_sum(acc[n][r]);
}

}  // namespace pk
}  // namespace talker_k

namespace talker_k {
namespace pk {

// ---- flag-carrying words: value in the low 32 bits, flag in the high 32 bits,
// written with one 8-byte store, so a reader that sees the flag sees the value.
__device__ __forceinline__ unsigned long long ll_pack(float v, uint32_t f) {
    return ((unsigned long long)f << 32) | __float_as_uint(v);
}
__device__ __forceinline__ void st_ll(unsigned long long *p, float v, uint32_t f) {
    asm volatile("st.volatile.global.u64 [%0], %1;" ::"l"(p), "l"(ll_pack(v, f)) : "memory");
}
__device__ __forceinline__ unsigned long long ld_ll(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.volatile.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void ld_ll2(const unsigned long long *p, unsigned long long &a, unsigned long long &b) {
    asm volatile("ld.volatile.global.v2.u64 {%0,%1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ uint32_t ll_flag(unsigned long long w) { return (uint32_t)(w >> 32); }
__device__ __forceinline__ float ll_val(unsigned long long w) { return __uint_as_float((uint32_t)w); }

// Re-read one word until its flag is f (bounded; returns at once after an abort).
// Sleeps between reads so that waiting threads leave issue slots and L1 bandwidth
// to the warps that are computing.
__device__ __noinline__ unsigned long long repoll_ll(const unsigned long long *p, uint32_t f, const Ctx &c) {
    unsigned long long w = ld_ll(p);
    if (ll_flag(w) == f || *c.abort_s) return w;
    const long long t0 = clock64();
    uint32_t ns = 32;
    for (uint32_t it = 1;; ++it) {
        __nanosleep(ns);
        if (ns < 256) ns <<= 1;
        w = ld_ll(p);
        if (ll_flag(w) == f) return w;
        if ((it & 15) == 0) {
            if (*c.abort_s || ld_volatile(c.abort_g)) {
                *c.abort_s = 1;
                return w;
            }
            if (clock64() - t0 > kWaitLimitCycles) {
                raise_abort(c);
                return w;
            }
        }
    }
}

// Bounded wait shared by the batch polls below: true once the caller should stop
// (grid abort seen, or the 1 s limit passed, which raises the abort).
__device__ __noinline__ bool poll_give_up(long long t0, const Ctx &c) {
    if (*c.abort_s || ld_volatile(c.abort_g)) {
        *c.abort_s = 1;
        return true;
    }
    if (clock64() - t0 > kWaitLimitCycles) {
        raise_abort(c);
        return true;
    }
    return false;
}

// Flags: one per (step, layer, tensor). base = step epoch * 256, never 0.
enum : uint32_t { FL_RAW = 0, FL_PART = 1, FL_O = 2, FL_X1 = 3, FL_ACT = 4, FL_X2 = 5 };
__device__ __forceinline__ uint32_t flag_of(uint32_t base, int layer, uint32_t what) {
    return base + (uint32_t)layer * 8u + what;
}

constexpr int KCAP = 3072;   // widest activation row the LL staging handles (R * KCAP / 2 pairs)

// Stage rows [0, rows) of a flag-word tensor (row stride ld words): every load
// is issued before any flag is checked, so a ready tensor costs one round trip.
// With `gain`, applies RMSNorm and the gain. Ends with a consumer barrier.
template <int EPV, int R>
__device__ void stage_ll(float *act, const unsigned long long *src, int ld, int K, int rows, uint32_t flag,
                         const float *gain, float eps, float *red, int ctid, const Ctx &c) {
    constexpr int NP = (R * KCAP / 2 + NCT - 1) / NCT;
    static_assert(NP <= 32, "stale mask holds 32 pairs");
    const int K2 = K >> 1;
    const int total = rows * K2;
    const int warp = ctid >> 5, lane = ctid & 31;
    unsigned long long wa[NP], wb[NP];
#pragma unroll
    for (int i = 0; i < NP; ++i) {
        const int idx = ctid + i * NCT;
        if (idx < total) {
            const int r = idx / K2, k = (idx - r * K2) * 2;
            ld_ll2(src + (size_t)r * ld + k, wa[i], wb[i]);
        }
    }
    float ss[R];
#pragma unroll
    for (int r = 0; r < R; ++r) ss[r] = 0.f;
    cbar();   // every warp is done reading the previous contents of act (the loads above are in flight)
    // Re-read every stale pair together, so that one polling round costs one round trip.
    uint32_t stale = 0;
#pragma unroll
    for (int i = 0; i < NP; ++i)
        if (ctid + i * NCT < total && (ll_flag(wa[i]) != flag || ll_flag(wb[i]) != flag)) stale |= 1u << i;
    if (stale != 0 && !*c.abort_s) {
        const long long t0 = clock64();
        for (uint32_t it = 1; stale != 0; ++it) {
            __nanosleep(64);
#pragma unroll
            for (int i = 0; i < NP; ++i)
                if (stale & (1u << i)) {
                    const int idx = ctid + i * NCT;
                    const int r = idx / K2, k = (idx - r * K2) * 2;
                    ld_ll2(src + (size_t)r * ld + k, wa[i], wb[i]);
                }
#pragma unroll
            for (int i = 0; i < NP; ++i)
                if ((stale & (1u << i)) && ll_flag(wa[i]) == flag && ll_flag(wb[i]) == flag) stale &= ~(1u << i);
            if (stale != 0 && (it & 15) == 0 && poll_give_up(t0, c)) break;
        }
    }
#pragma unroll
    for (int i = 0; i < NP; ++i) {
        const int idx = ctid + i * NCT;
        if (idx < total) {
            const int r = idx / K2, k = (idx - r * K2) * 2;
            const float v0 = ll_val(wa[i]), v1 = ll_val(wb[i]);
            act[aidx<EPV>(r, k, K)] = v0;
            act[aidx<EPV>(r, k + 1, K)] = v1;
            const float s2 = v0 * v0 + v1 * v1;
#pragma unroll
            for (int rr = 0; rr < R; ++rr)
                if (rr == r) ss[rr] += s2;
        }
    }
    if (gain != nullptr) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float v = warp_sum(ss[r]);
            if (lane == 0) red[warp * R + r] = v;
        }
        cbar();
        float inv[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float t = 0.f;
            for (int w = 0; w < NCW; ++w) t += red[w * R + r];
            inv[r] = 1.0f / sqrtf(t / (float)K + eps);
        }
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            const int idx = ctid + i * NCT;
            if (idx < total) {
                const int r = idx / K2, k = (idx - r * K2) * 2;
                float iv = inv[0];
#pragma unroll
                for (int rr = 1; rr < R; ++rr)
                    if (rr == r) iv = inv[rr];
                float *a0 = act + aidx<EPV>(r, k, K);
                float *a1 = act + aidx<EPV>(r, k + 1, K);
                *a0 = *a0 * iv * gain[k];
                *a1 = *a1 * iv * gain[k + 1];
            }
        }
    }
    cbar();
}

}  // namespace pk
}  // namespace talker_k

namespace talker_k {
namespace pk {

template <int R>
__device__ __forceinline__ float pick(const float (&a)[R], int r) {
    float v = a[0];
#pragma unroll
    for (int i = 1; i < R; ++i)
        if (i == r) v = a[i];
    return v;
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

constexpr int XO = 64;   // owned residual rows per CTA (ceil(H / grid) <= XO)

template <typename WT, typename KT, int HD, int R>
__global__ void __launch_bounds__(NT, 1) k_decode_persistent(const PersistParams p) {
    constexpr int EPV = Elem<WT>::kPerVec;
    constexpr size_t WSZ = sizeof(WT);
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ __align__(8) uint64_t full[NS], empty[NS];
    __shared__ float red[NCW * R];
    __shared__ float m_s[MAXG], l_s[MAXG], al_s[MAXG];
    __shared__ float ml_s[MAXG][kMaxSplits][2];
    __shared__ float xown[R][XO];
    __shared__ float bv_s[NCW][R];
    __shared__ int bi_s[NCW][R];
    __shared__ int curlen_s[R];
    __shared__ int abort_sh, flag_s;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int P = gridDim.x, cta = blockIdx.x;
    const int H = p.H, half = HD / 2, G = p.G;
    const int qd = p.nq * HD, qkv_n = (p.nq + 2 * p.nkv) * HD;
    const int KMAX = max(max(H, qd), p.I);
    const int rows = p.rows;
    unsigned char *ring = smem;
    float *act = reinterpret_cast<float *>(smem + (size_t)NS * SLOT);
    float *qs = act + (size_t)R * KMAX;            // [G][HD] scaled q of the attention row
    float *sc = qs + MAXG * HD;                     // [G][kPage] scores / probabilities
    KT *knew = reinterpret_cast<KT *>(sc + MAXG * kPage);
    KT *vnew = knew + HD;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NCW);
        }
        abort_sh = 0;
        fence_barrier_init();
    }
    if (tid < R) curlen_s[tid] = (tid < rows) ? p.cur_len[tid] : 0;
    __syncthreads();
    const Ctx c{reinterpret_cast<volatile int *>(&abort_sh), p.sync + SY_ABORT, p.status};
    const AttnWork aw = attn_work(p, cta, P, curlen_s);

    if (warp == NCW) {
        if (lane == 0) producer<WT, KT, HD>(p, ring, full, empty, c, aw);
        return;
    }

    // ------------------------------------------------------------------ consumers
    const int ctid = tid;
    unsigned long long *trace = (p.trace != nullptr && ctid == 0) ? p.trace + (size_t)cta * kTraceSlots : nullptr;
    if (trace) {   // clock64 stamps; this pair aligns them across CTAs
        trace[kTraceSlots - 2] = globaltimer_ns();
        trace[kTraceSlots - 1] = clock64();
    }
    Ring rc{ring, full, empty, 0, trace};
#define TR(slot)                                      \
    do {                                              \
        if (trace) trace[(slot)] = clock64();         \
    } while (0)
    const Span own = cta_span(H, cta, P);           // residual rows this CTA updates (o_proj and down)
    for (int i = ctid; i < rows * own.n; i += NCT) {
        const int r = i / own.n, j = i - r * own.n;
        xown[r][j] = p.emb[(size_t)r * H + own.u0 + j];
    }

    for (int l = 0; l < p.n_layers; ++l) {
        const LayerW &L = p.layers[l];
        const int tb = l * kTracePerLayer;
        TR(tb + 0);
        // ---- RMSNorm -> [Wq;Wk;Wv] -> raw q|k|v words
        // (A CTA with no rows in a phase skips that phase's input: it would have no
        // output that orders its reads before the next overwrite of the input words.)
        const Span sq = cta_span(qkv_n, cta, P);
        if (sq.n > 0) {
            if (l == 0) stage<EPV, R>(act, p.emb, H, H, rows, L.in_norm, p.eps, red, ctid);
            else stage_ll<EPV, R>(act, p.x_ll, H, H, rows, flag_of(p.flag_base, l - 1, FL_X2), L.in_norm, p.eps,
                                  red, ctid, c);
        }
        TR(tb + 1);
        {
            const uint32_t f = flag_of(p.flag_base, l, FL_RAW);
            const Span s = sq;
            const int upc = max(1, (int)(SLOT / (H * WSZ)));
            for (int u = s.u0; u < s.u0 + s.n; u += upc) {
                const int n = min(upc, s.u0 + s.n - u);
                const unsigned char *w = rc.acquire(c);
                for (int j = warp; j < n; j += NCW) {
                    float acc[1][R];
                    dot_rows<WT, R, 1>(w + (size_t)j * H * WSZ, H, act, rows, acc, lane);
                    if (lane < rows) st_ll(p.raw_ll + (size_t)lane * qkv_n + u + j, pick<R>(acc[0], lane), f);
                }
                rc.release(lane);
            }
        }
        TR(tb + 2);
        // ---- attention of (row r, KV group g, split) over [0, pos]
        if (aw.has) {
            const int r = aw.r, g = aw.g, pos = aw.pos;
            if (warp < G + 2) {
                // QK-norm + RoPE of this row's q heads of the group and k; v as is
                const int h = (warp < G) ? g * G + warp : (warp == G ? p.nq + g : p.nq + p.nkv + g);
                const unsigned long long *src = p.raw_ll + (size_t)r * qkv_n + (size_t)h * HD;
                const uint32_t f = flag_of(p.flag_base, l, FL_RAW);
                unsigned long long wv[4];
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const int i = lane + 32 * t;
                    if (i < half) {
                        wv[2 * t] = ld_ll(src + i);
                        wv[2 * t + 1] = ld_ll(src + i + half);
                    }
                }
                // word 2t + u sits at src + lane + 32t + u * half; stale words are re-read together
                uint32_t stale = 0;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (lane + 32 * (q >> 1) < half && ll_flag(wv[q]) != f) stale |= 1u << q;
                if (stale != 0 && !*c.abort_s) {
                    const long long t0 = clock64();
                    for (uint32_t it = 1; stale != 0; ++it) {
                        __nanosleep(64);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if (stale & (1u << q)) wv[q] = ld_ll(src + lane + 32 * (q >> 1) + (q & 1) * half);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if ((stale & (1u << q)) && ll_flag(wv[q]) == f) stale &= ~(1u << q);
                        if (stale != 0 && (it & 15) == 0 && poll_give_up(t0, c)) break;
                    }
                }
                float a[2], b[2];
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const int i = lane + 32 * t;
                    a[t] = b[t] = 0.f;
                    if (i < half) {
                        a[t] = ll_val(wv[2 * t]);
                        b[t] = ll_val(wv[2 * t + 1]);
                    }
                }
                if (warp <= G) {
                    const float *gain = (warp < G) ? L.q_norm : L.k_norm;
                    const float ss = warp_sum(a[0] * a[0] + b[0] * b[0] + a[1] * a[1] + b[1] * b[1]);
                    const float inv = 1.0f / sqrtf(ss / (float)HD + p.eps);
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        const int i = lane + 32 * t;
                        if (i < half) {
                            const float x0 = a[t] * inv * gain[i], x1 = b[t] * inv * gain[i + half];
                            const float2 cs = p.rope[(size_t)pos * half + i];
                            a[t] = x0 * cs.x - x1 * cs.y;
                            b[t] = x1 * cs.x + x0 * cs.y;
                        }
                    }
                }
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const int i = lane + 32 * t;
                    if (i >= half) continue;
                    if (warp < G) {
                        qs[warp * HD + i] = a[t] * p.scale;
                        qs[warp * HD + i + half] = b[t] * p.scale;
                    } else {
                        KT *d = (warp == G) ? knew : vnew;
                        Elem<KT>::store(d, i, a[t]);
                        Elem<KT>::store(d, i + half, b[t]);
                        if (aw.split == 0) {   // the cache keeps this row for later steps
                            const int page = p.cache.page_table[(size_t)r * p.cache.pages_per_stream + pos / kPage];
                            const size_t off = (size_t)page * p.cache.page_elems +
                                               ((size_t)(l * p.cache.n_kv + g) * kPage + pos % kPage) * HD;
                            KT *cp = static_cast<KT *>(warp == G ? p.cache.k : p.cache.v) + off;
                            Elem<KT>::store(cp, i, a[t]);
                            Elem<KT>::store(cp, i + half, b[t]);
                        }
                    }
                }
            }
            if (ctid < G) {
                m_s[ctid] = -INFINITY;
                l_s[ctid] = 0.f;
            }
            constexpr int NO = (MAXG * HD + NCT - 1) / NCT;
            float o_acc[NO];
#pragma unroll
            for (int o = 0; o < NO; ++o) o_acc[o] = 0.f;
            cbar();
            TR(tb + 3);
            for (int pg = aw.pb; pg < aw.pe; ++pg) {
                KT *Ks = reinterpret_cast<KT *>(const_cast<unsigned char *>(rc.acquire(c)));
                KT *Vs = Ks + kPage * HD;
                const int valid = min(kPage, pos + 1 - pg * kPage);
                if (pg == pos / kPage) {   // this step's row is not in the cached copy yet
                    for (int i = ctid; i < HD; i += NCT) {
                        Ks[(pos % kPage) * HD + i] = knew[i];
                        Vs[(pos % kPage) * HD + i] = vnew[i];
                    }
                    fence_proxy_async();   // generic writes into a slot that a later bulk copy refills
                    cbar();
                }
                // Scores: each warp takes rows j = warp + NCW * i, loads all of them first,
                // forms every (row, head) partial dot, then reduces them in one interleaved
                // butterfly, so the shuffle latency is paid once per warp, not per row.
                constexpr int E = HD / 32;
                constexpr int RPW = (kPage + NCW - 1) / NCW;   // rows per warp
                float kv[RPW][E];
#pragma unroll
                for (int i = 0; i < RPW; ++i) {
                    const int j = warp + NCW * i;
#pragma unroll
                    for (int e = 0; e < E; ++e)
                        kv[i][e] = (j < kPage) ? Elem<KT>::load(Ks, (size_t)j * HD + lane * E + e) : 0.f;
                }
                float qv[MAXG][E];
#pragma unroll
                for (int gi = 0; gi < MAXG; ++gi)
#pragma unroll
                    for (int e = 0; e < E; ++e) qv[gi][e] = (gi < G) ? qs[gi * HD + lane * E + e] : 0.f;
                float dv[RPW][MAXG];
#pragma unroll
                for (int i = 0; i < RPW; ++i)
#pragma unroll
                    for (int gi = 0; gi < MAXG; ++gi) {
                        float d = 0.f;
#pragma unroll
                        for (int e = 0; e < E; ++e) d = fmaf(qv[gi][e], kv[i][e], d);
                        dv[i][gi] = d;
                    }
                if (G == 2) {
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                        for (int i = 0; i < RPW; ++i) {
                            dv[i][0] += __shfl_xor_sync(0xffffffffu, dv[i][0], o);
                            dv[i][1] += __shfl_xor_sync(0xffffffffu, dv[i][1], o);
                        }
                } else {
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                        for (int i = 0; i < RPW; ++i)
#pragma unroll
                            for (int gi = 0; gi < MAXG; ++gi)
                                if (gi < G) dv[i][gi] += __shfl_xor_sync(0xffffffffu, dv[i][gi], o);
                }
                if (lane == 0) {
#pragma unroll
                    for (int i = 0; i < RPW; ++i) {
                        const int j = warp + NCW * i;
                        if (j < kPage)
#pragma unroll
                            for (int gi = 0; gi < MAXG; ++gi)
                                if (gi < G) sc[gi * kPage + j] = (j < valid) ? dv[i][gi] : -INFINITY;
                    }
                }
                cbar();
                if (warp < G) {
                    const int gi = warp;
                    const float v0 = sc[gi * kPage + lane], v1 = sc[gi * kPage + lane + 32];
                    const float m_old = m_s[gi];
                    const float m_new = fmaxf(m_old, warp_max(fmaxf(v0, v1)));
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
                cbar();
#pragma unroll
                for (int o = 0; o < NO; ++o) {
                    const int idx = ctid + o * NCT;
                    if (idx < G * HD) {
                        const int gi = idx / HD, d = idx - gi * HD;
                        float acc = o_acc[o] * al_s[gi];
                        const float *pj = sc + gi * kPage;
                        for (int j = 0; j < valid; ++j) acc = fmaf(pj[j], Elem<KT>::load(Vs, (size_t)j * HD + d), acc);
                        o_acc[o] = acc;
                    }
                }
                rc.release(lane);
                cbar();
            }
            TR(tb + 5);
            const int hq0 = g * G;
            unsigned long long *orow = p.o_ll + (size_t)r * qd;
            const uint32_t fo = flag_of(p.flag_base, l, FL_O);
            constexpr int WS = HD + 2;
            if (aw.nact == 1) {
#pragma unroll
                for (int o = 0; o < NO; ++o) {
                    const int idx = ctid + o * NCT;
                    if (idx < G * HD) {
                        const int gi = idx / HD, d = idx - gi * HD;
                        st_ll(orow + (hq0 + gi) * HD + d, o_acc[o] / l_s[gi], fo);
                    }
                }
            } else if (aw.split != 0) {
                // publish this split's (m, l, o) for the combining CTA (split 0)
                const uint32_t fp = flag_of(p.flag_base, l, FL_PART);
#pragma unroll
                for (int o = 0; o < NO; ++o) {
                    const int idx = ctid + o * NCT;
                    if (idx < G * HD) {
                        const int gi = idx / HD, d = idx - gi * HD;
                        unsigned long long *w =
                            p.part_ll + (((size_t)r * p.nq + hq0 + gi) * kMaxSplits + aw.split) * WS;
                        st_ll(w + 2 + d, o_acc[o], fp);
                        if (d == 0) {
                            st_ll(w, m_s[gi], fp);
                            st_ll(w + 1, l_s[gi], fp);
                        }
                    }
                }
            } else {
                // split 0 combines all splits in split order (deterministic)
                const uint32_t fp = flag_of(p.flag_base, l, FL_PART);
                const int ns = aw.nact;
                // Issue this thread's o loads of every split first (all in flight together),
                // then gather (m, l) of splits 1..ns-1 into shared memory.
                auto gather_o = [&](int idx, float (&ov)[kMaxSplits]) {
                    const int gi = idx / HD, d = idx - gi * HD;
                    const unsigned long long *wb =
                        p.part_ll + (((size_t)r * p.nq + hq0 + gi) * kMaxSplits) * WS + 2 + d;
                    unsigned long long wv2[kMaxSplits];
#pragma unroll
                    for (int sp = 1; sp < kMaxSplits; ++sp)
                        if (sp < ns) wv2[sp] = ld_ll(wb + (size_t)sp * WS);
                    uint32_t stale = 0;
#pragma unroll
                    for (int sp = 1; sp < kMaxSplits; ++sp)
                        if (sp < ns && ll_flag(wv2[sp]) != fp) stale |= 1u << sp;
                    if (stale != 0 && !*c.abort_s) {
                        const long long t0 = clock64();
                        for (uint32_t it = 1; stale != 0; ++it) {
                            __nanosleep(64);
#pragma unroll
                            for (int sp = 1; sp < kMaxSplits; ++sp)
                                if (stale & (1u << sp)) wv2[sp] = ld_ll(wb + (size_t)sp * WS);
#pragma unroll
                            for (int sp = 1; sp < kMaxSplits; ++sp)
                                if ((stale & (1u << sp)) && ll_flag(wv2[sp]) == fp) stale &= ~(1u << sp);
                            if (stale != 0 && (it & 15) == 0 && poll_give_up(t0, c)) break;
                        }
                    }
#pragma unroll
                    for (int sp = 1; sp < kMaxSplits; ++sp) ov[sp] = (sp < ns) ? ll_val(wv2[sp]) : 0.f;
                };
                auto combine_o = [&](int idx, float own_o, float (&ov)[kMaxSplits]) {
                    const int gi = idx / HD, d = idx - gi * HD;
                    ov[0] = own_o;
                    float M = -INFINITY;
                    for (int sp = 0; sp < ns; ++sp) M = fmaxf(M, ml_s[gi][sp][0]);
                    float Ls = 0.f, O = 0.f;
#pragma unroll
                    for (int sp = 0; sp < kMaxSplits; ++sp)
                        if (sp < ns) {
                            const float f = expf(ml_s[gi][sp][0] - M);
                            Ls = fmaf(ml_s[gi][sp][1], f, Ls);
                            O = fmaf(ov[sp], f, O);
                        }
                    st_ll(orow + (hq0 + gi) * HD + d, O / Ls, fo);
                };
                float ov[kMaxSplits];
                if (ctid < G * HD) gather_o(ctid, ov);
                for (int idx = ctid; idx < G * (ns - 1) * 2; idx += NCT) {
                    const int gi = idx / ((ns - 1) * 2), rem = idx - gi * (ns - 1) * 2;
                    const int sp = 1 + rem / 2, which = rem & 1;
                    const unsigned long long *w =
                        p.part_ll + (((size_t)r * p.nq + hq0 + gi) * kMaxSplits + sp) * WS + which;
                    unsigned long long v = ld_ll(w);
                    if (ll_flag(v) != fp) v = repoll_ll(w, fp, c);
                    ml_s[gi][sp][which] = ll_val(v);
                }
                if (ctid < G) {
                    ml_s[ctid][0][0] = m_s[ctid];
                    ml_s[ctid][0][1] = l_s[ctid];
                }
                cbar();
                TR(tb + 8);
                if (ctid < G * HD) combine_o(ctid, o_acc[0], ov);
#pragma unroll
                for (int o = 1; o < NO; ++o) {
                    const int idx = ctid + o * NCT;
                    if (idx < G * HD) {
                        gather_o(idx, ov);
                        combine_o(idx, o_acc[o], ov);
                    }
                }
            }
        }
        TR(tb + 4);

        // ---- o_proj + residual
        if (own.n > 0)
            stage_ll<EPV, R>(act, p.o_ll, qd, qd, rows, flag_of(p.flag_base, l, FL_O), nullptr, 0.f, red, ctid, c);
        TR(tb + 6);
        {
            const uint32_t f = flag_of(p.flag_base, l, FL_X1);
            const int upc = max(1, (int)(SLOT / (qd * WSZ)));
            for (int u = own.u0; u < own.u0 + own.n; u += upc) {
                const int n = min(upc, own.u0 + own.n - u);
                const unsigned char *w = rc.acquire(c);
                for (int j = warp; j < n; j += NCW) {
                    float acc[1][R];
                    dot_rows<WT, R, 1>(w + (size_t)j * qd * WSZ, qd, act, rows, acc, lane);
                    if (lane < rows) {
                        const int jj = u + j - own.u0;
                        const float x1 = xown[lane][jj] + pick<R>(acc[0], lane);
                        xown[lane][jj] = x1;
                        st_ll(p.x_ll + (size_t)lane * H + u + j, x1, f);
                    }
                }
                rc.release(lane);
            }
        }
        TR(tb + 7);

        // ---- post-norm -> [Wg;Wu] -> silu(gate) * up
        const Span sg = cta_span(p.I, cta, P);
        if (sg.n > 0)
            stage_ll<EPV, R>(act, p.x_ll, H, H, rows, flag_of(p.flag_base, l, FL_X1), L.post_norm, p.eps, red, ctid,
                             c);
        TR(tb + 9);
        {
            const uint32_t f = flag_of(p.flag_base, l, FL_ACT);
            const Span s = sg;
            const int upc = max(1, (int)(SLOT / (2 * H * WSZ)));
            for (int u = s.u0; u < s.u0 + s.n; u += upc) {
                const int n = min(upc, s.u0 + s.n - u);
                const unsigned char *w = rc.acquire(c);
                for (int j = warp; j < n; j += NCW) {
                    float acc[2][R];
                    dot_rows<WT, R, 2>(w + (size_t)j * 2 * H * WSZ, H, act, rows, acc, lane);
                    if (lane < rows)
                        st_ll(p.act_ll + (size_t)lane * p.I + u + j,
                              silu_f(pick<R>(acc[0], lane)) * pick<R>(acc[1], lane), f);
                }
                rc.release(lane);
            }
        }
        TR(tb + 10);

        // ---- down + residual
        if (own.n > 0)
            stage_ll<EPV, R>(act, p.act_ll, p.I, p.I, rows, flag_of(p.flag_base, l, FL_ACT), nullptr, 0.f, red, ctid,
                             c);
        TR(tb + 12);
        {
            const uint32_t f = flag_of(p.flag_base, l, FL_X2);
            const int upc = max(1, (int)(SLOT / (p.I * WSZ)));
            for (int u = own.u0; u < own.u0 + own.n; u += upc) {
                const int n = min(upc, own.u0 + own.n - u);
                const unsigned char *w = rc.acquire(c);
                for (int j = warp; j < n; j += NCW) {
                    float acc[1][R];
                    dot_rows<WT, R, 1>(w + (size_t)j * p.I * WSZ, p.I, act, rows, acc, lane);
                    if (lane < rows) {
                        const int jj = u + j - own.u0;
                        const float x2 = xown[lane][jj] + pick<R>(acc[0], lane);
                        xown[lane][jj] = x2;
                        st_ll(p.x_ll + (size_t)lane * H + u + j, x2, f);
                    }
                }
                rc.release(lane);
            }
        }
        TR(tb + 13);
    }

    // ---- final norm -> codec_head -> logits, hidden, argmax
    const int th = p.n_layers * kTracePerLayer;
    stage_ll<EPV, R>(act, p.x_ll, H, H, rows, flag_of(p.flag_base, p.n_layers - 1, FL_X2), p.final_norm, p.eps, red,
                     ctid, c);
    TR(th + 0);
    if (cta == 0 && p.hidden_out != nullptr)
        for (int i = ctid; i < rows * H; i += NCT) {
            const int r = i / H, k = i - r * H;
            p.hidden_out[i] = act[aidx<EPV>(r, k, H)];
        }
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    {
        const Span s = cta_span(p.V, cta, P);
        const int upc = max(1, (int)(SLOT / (H * WSZ)));
        for (int u = s.u0; u < s.u0 + s.n; u += upc) {
            const int n = min(upc, s.u0 + s.n - u);
            const unsigned char *w = rc.acquire(c);
            for (int j = warp; j < n; j += NCW) {
                float acc[1][R];
                dot_rows<WT, R, 1>(w + (size_t)j * H * WSZ, H, act, rows, acc, lane);
                if (lane < rows) {
                    const float v = pick<R>(acc[0], lane);
                    p.logits[(size_t)lane * p.V + u + j] = v;
                    if (isnan(v)) atomicOr(p.status, ST_NAN_LOGIT);
                    else if (v > bv || (v == bv && u + j < bi)) {
                        bv = v;
                        bi = u + j;
                    }
                }
            }
            rc.release(lane);
        }
    }
    TR(th + 1);
    if (lane < R) {
        bv_s[warp][lane] = bv;
        bi_s[warp][lane] = bi;
    }
    cbar();
    if (ctid < rows) {
        float b = -INFINITY;
        int ib = 0x7fffffff;
        for (int w = 0; w < NCW; ++w) {
            const float v = bv_s[w][ctid];
            const int i = bi_s[w][ctid];
            if (v > b || (v == b && i < ib)) {
                b = v;
                ib = i;
            }
        }
        p.head_val[(size_t)cta * 4 + ctid] = b;
        p.head_idx[(size_t)cta * 4 + ctid] = ib;
    }
    __threadfence();
    cbar();
    if (ctid == 0) flag_s = (atomicAdd(p.sync + SY_HEAD, 1) == P - 1);
    cbar();
    if (flag_s) {
        __threadfence();
        // each row is reduced by 4 warps (128 threads), then across those warps
        const int r = warp >> 2, sub = ctid & 127;
        float b = -INFINITY;
        int ib = 0x7fffffff;
        if (r < rows) {
            for (int s2 = sub; s2 < P; s2 += 128) {
                const float v = __ldcg(p.head_val + (size_t)s2 * 4 + r);
                const int i = __ldcg(p.head_idx + (size_t)s2 * 4 + r);
                if (v > b || (v == b && i < ib)) {
                    b = v;
                    ib = i;
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float v2 = __shfl_xor_sync(0xffffffffu, b, o);
            const int i2 = __shfl_xor_sync(0xffffffffu, ib, o);
            if (v2 > b || (v2 == b && i2 < ib)) {
                b = v2;
                ib = i2;
            }
        }
        if (lane == 0) {
            bv_s[warp][0] = b;
            bi_s[warp][0] = ib;
        }
        cbar();
        if (ctid < rows) {
            float bb = -INFINITY;
            int ii = 0x7fffffff;
            for (int w = 4 * ctid; w < min(4 * ctid + 4, NCW); ++w) {
                if (bv_s[w][0] > bb || (bv_s[w][0] == bb && bi_s[w][0] < ii)) {
                    bb = bv_s[w][0];
                    ii = bi_s[w][0];
                }
            }
            if (p.argmax_out != nullptr) p.argmax_out[ctid] = ii;
            p.cur_len[ctid] = curlen_s[ctid] + 1;
        }
        if (ctid == 0) {
            p.sync[SY_HEAD] = 0;     // every CTA has arrived: ready for the next launch
            p.sync[SY_ABORT] = 0;
        }
    }
    TR(th + 2);
#undef TR
}

size_t persist_smem_bytes(int R, int head_dim, int kv_bf16, int kmax) {
    return (size_t)NS * SLOT + (size_t)R * kmax * 4 + (size_t)MAXG * head_dim * 4 + (size_t)MAXG * kPage * 4 +
           2 * (size_t)head_dim * (kv_bf16 ? 2 : 4) + 16;
}

}  // namespace pk
}  // namespace talker_k
namespace talker_k {

template <typename WT, typename KT, int HD, int R>
static cudaError_t launch_pk(const PersistParams &p, int grid, size_t smem, cudaStream_t st) {
    void *args[] = {const_cast<PersistParams *>(&p)};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(pk::k_decode_persistent<WT, KT, HD, R>), grid,
                                       pk::NT, args, smem, st);
}

template <typename WT, typename KT, int HD, int R>
static cudaError_t setup_pk(size_t smem, int *blocks_per_sm) {
    const void *f = reinterpret_cast<const void *>(pk::k_decode_persistent<WT, KT, HD, R>);
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, f, pk::NT, smem);
}

#define PK_DISPATCH(FN, ...)                                                                 \
    do {                                                                                     \
        const int key = (w_bf16 ? 1000 : 0) + head_dim * 10 + R;                             \
        switch (key) {                                                                       \
            case 321: return FN<float, float, 32, 1>(__VA_ARGS__);                           \
            case 324: return FN<float, float, 32, 4>(__VA_ARGS__);                           \
            case 641: return FN<float, float, 64, 1>(__VA_ARGS__);                           \
            case 644: return FN<float, float, 64, 4>(__VA_ARGS__);                           \
            case 1281: return FN<float, float, 128, 1>(__VA_ARGS__);                         \
            case 1284: return FN<float, float, 128, 4>(__VA_ARGS__);                         \
            case 1321: return FN<__nv_bfloat16, __nv_bfloat16, 32, 1>(__VA_ARGS__);         \
            case 1324: return FN<__nv_bfloat16, __nv_bfloat16, 32, 4>(__VA_ARGS__);         \
            case 1641: return FN<__nv_bfloat16, __nv_bfloat16, 64, 1>(__VA_ARGS__);         \
            case 1644: return FN<__nv_bfloat16, __nv_bfloat16, 64, 4>(__VA_ARGS__);         \
            case 2281: return FN<__nv_bfloat16, __nv_bfloat16, 128, 1>(__VA_ARGS__);        \
            case 2284: return FN<__nv_bfloat16, __nv_bfloat16, 128, 4>(__VA_ARGS__);        \
        }                                                                                    \
        return cudaErrorInvalidValue;                                                        \
    } while (0)

size_t persist_smem(int R, int head_dim, int kv_bf16, int kmax, int group, int splits) {
    (void)group;
    (void)splits;
    return pk::persist_smem_bytes(R, head_dim, kv_bf16, kmax);
}
int persist_threads() { return pk::NT; }
int persist_slot_bytes() { return pk::SLOT; }
int persist_sync_words(int n_heads) { return pk::SY_ROWS + n_heads; }

cudaError_t setup_persistent(int w_bf16, int head_dim, int R, size_t smem, int *blocks_per_sm) {
    PK_DISPATCH(setup_pk, smem, blocks_per_sm);
}

cudaError_t launch_persistent(int w_bf16, int head_dim, int R, const PersistParams &p, int grid, size_t smem,
                              cudaStream_t st) {
    PK_DISPATCH(launch_pk, p, grid, smem, st);
}

}  // namespace talker_k
