// Host runtime of the C-ABI declared in include/talker.h: weight store,
// paged KV cache, workspaces, per-stream length bookkeeping, kernel sequencing
// and the replayed CUDA graph of a decode step.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <vector>

#include "kernels.cuh"
#include "talker.h"

using namespace talker_k;

namespace {

constexpr int kPageRows = 64;     // positions per KV page (kernels use the same constant)
constexpr int kMaxGraphs = 8;     // cached decode graphs per handle

struct LayerDev {
    const float *in_norm, *post_norm, *q_norm, *k_norm;
    const void *qkv, *o, *gu, *down;
};

// A captured prefill (or batched prefill): replayed while every input of the key is the same.
struct PrefillGraph {
    std::vector<long long> key;
    cudaGraphExec_t exec;
    int n_kernels;
};

struct GraphEntry {
    int kind;   // 0: GEMV kernels, 1: tensor-core GEMMs
    int B;
    int splits, cluster;   // attention splits per (row, KV group); 1: splits combine inside a cluster
    int mm;                // attention on the tensor cores (bf16 tiles through the tensor maps)
    const float *emb;
    float *logits, *hidden;
    int32_t *argmax;
    const int32_t *ids;     // codebook ids of a step whose input rows are gathered (else null)
    const float *overlay;
    cudaGraphExec_t exec;
    int n_kernels;
};

thread_local char g_last_error[256] = "";

talker_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return TALKER_OK;
    snprintf(g_last_error, sizeof(g_last_error), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
    cudaGetLastError();  // clear a non-sticky error so the handle stays usable
    return e == cudaErrorMemoryAllocation ? TALKER_ENOMEM : TALKER_ECUDA;
}

#define TRY_CUDA(expr)                                     \
    do {                                                   \
        cudaError_t e_ = (expr);                           \
        if (e_ != cudaSuccess) return from_cuda(e_);       \
    } while (0)

#define TRY(expr)                                          \
    do {                                                   \
        talker_status s_ = (expr);                         \
        if (s_ != TALKER_OK) return s_;                    \
    } while (0)

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace

struct talker {
    talker_config c{};
    cudaStream_t st = nullptr;
    cudaStream_t cap_st = nullptr;  // private stream for graph capture (the caller's may be the legacy stream)
    int dev = 0, n_sm = 0;
    int H = 0, nq = 0, nkv = 0, hd = 0, qd = 0, kvd = 0, qkv_n = 0, I = 0, V = 0, G = 0;
    int w_bf16 = 0, kv_bf16 = 0, kv_q8 = 0, kv_kind = 0;   // kv_kind: 0 f32, 1 bf16, 2 Q8_0
    size_t wsz = 0, kvsz = 0;
    char *wstore = nullptr;
    std::vector<LayerDev> L;
    const float *fnorm = nullptr;
    const void *head = nullptr;
    // KV cache
    int n_streams = 0, max_seq = 0, pps = 0;
    size_t page_elems = 0;
    KvMaps kv_maps{};                    // tensor maps of the bf16 pools (head_dim 128)
    bool kv_maps_ok = false;
    void *kpool = nullptr, *vpool = nullptr;
    int *d_pt = nullptr, *d_len = nullptr;
    float2 *d_rope = nullptr;
    std::vector<int> len;
    // activations, sized for cap_rows rows
    int cap_rows = 0;
    float *x = nullptr, *raw = nullptr, *q = nullptr, *attn = nullptr, *act = nullptr;
    float *x2 = nullptr;   // GEMV decode with the fused MLP: the residual stream (x: its post-attention copy)
    // workspaces
    size_t cap_attn_ws = 0, cap_head_part = 0;
    float *attn_ws = nullptr, *head_val = nullptr;
    int *head_idx = nullptr;
    int cap_cnt_rows = 0;
    int *qkv_cnt = nullptr, *attn_cnt = nullptr, *head_cnt = nullptr;
    int *d_status = nullptr;
    int64_t launches = 0;
    std::vector<GraphEntry> graphs;
    std::vector<PrefillGraph> pgraphs;
    int decode_mode = 0;                 // 0 auto, 2 GEMV graph, 3 tensor-core graph
    int attn_cluster = 0;   // decode attention: splits combine inside a thread-block cluster
    int attn_mm = 0;        // decode attention: bf16 tiles through the tensor maps, tensor-core scores and P.V
    int prefill_mode = 0;                // 0 automatic, 2 always the GEMV kernels, 3 / 4 tensor-core GEMMs
                                         // with the mma.sync / the tcgen05 attention at any T
    // tensor-core prefill buffers (bf16 GEMM operands and the f32 gate/up projection)
    int cap_tc_rows = 0;
    int cap_kd_keys = 0;                 // keys kd_tc / vt_tc hold per KV head
    void *hb = nullptr, *ab = nullptr, *gb = nullptr;
    __nv_bfloat16 *kv_dense = nullptr;   // Q8_0 storage: the prefill's own k / v rows, [2][rows][n_kv][hd]
    __nv_bfloat16 *kd_tc = nullptr;      // tcgen05 prefill attention: K [n_kv][L][hd] and V^T [n_kv][hd][L]
    __nv_bfloat16 *vt_tc = nullptr;
    float *gu = nullptr;                 // split-K [gate; up] sums: all zeros between uses
    int *gemm_cnt = nullptr;             // per-tile split counters of the split-K SwiGLU GEMM: zeros between uses
    int tc_ok = -1;                      // tensor-core prefill usable for this geometry (-1 unknown)
    // TTS loop input / output
    int suppress_tail = 0, suppress_eos = -1;   // head: logits [V - tail, V) except eos become -inf
    std::vector<const void *> code_tables;      // caller-owned codebook tables (empty: none)
    std::vector<int> code_vocab;
    int code_bf16 = 0;
    const void **d_code_tables = nullptr;       // device copies of the table pointers and vocab sizes,
    int *d_code_vocab = nullptr;                // read by the kernels that gather input rows
    // whole-frame graph (prefill + steps fed by the previous step's code, on the device)
    cudaGraphExec_t frame_exec = nullptr;
    std::vector<const void *> frame_key;        // the inputs the captured frame is valid for
    int frame_T0 = 0, frame_steps = 0, frame_kernels = 0;
    float *frame_logits = nullptr;              // [V] scratch when the caller wants no logits
};

namespace {

void drop_graphs(talker *t) {
    for (auto &g : t->graphs) cudaGraphExecDestroy(g.exec);
    t->graphs.clear();
    for (auto &g : t->pgraphs) cudaGraphExecDestroy(g.exec);
    t->pgraphs.clear();
    if (t->frame_exec) cudaGraphExecDestroy(t->frame_exec);
    t->frame_exec = nullptr;
    t->frame_key.clear();
}

void free_ptr(void *p) {
    if (p) cudaFree(p);
}

void free_workspaces(talker *t) {
    float **fl[] = {&t->x, &t->raw, &t->q, &t->attn, &t->act, &t->attn_ws, &t->head_val, &t->frame_logits,
                    &t->x2};
    for (auto pp : fl) {
        free_ptr(*pp);
        *pp = nullptr;
    }
    int **il[] = {&t->head_idx, &t->qkv_cnt, &t->attn_cnt, &t->head_cnt};
    for (auto pp : il) {
        free_ptr(*pp);
        *pp = nullptr;
    }
    t->cap_rows = 0;
    t->cap_attn_ws = t->cap_head_part = 0;
    t->cap_cnt_rows = 0;
}

void free_tc(talker *t) {
    void **bl[] = {&t->hb, &t->ab, &t->gb, reinterpret_cast<void **>(&t->gu), reinterpret_cast<void **>(&t->kv_dense),
                   reinterpret_cast<void **>(&t->kd_tc), reinterpret_cast<void **>(&t->vt_tc),
                   reinterpret_cast<void **>(&t->gemm_cnt)};
    for (auto pp : bl) {
        free_ptr(*pp);
        *pp = nullptr;
    }
    t->cap_tc_rows = 0;
    t->cap_kd_keys = 0;
}

void free_cache(talker *t) {
    free_ptr(t->kpool);
    free_ptr(t->vpool);
    free_ptr(t->d_pt);
    free_ptr(t->d_len);
    free_ptr(t->d_rope);
    t->kpool = t->vpool = nullptr;
    t->d_pt = t->d_len = nullptr;
    t->d_rope = nullptr;
    t->kv_maps_ok = false;
    t->n_streams = t->max_seq = t->pps = 0;
    t->len.clear();
}

// Row-block height of the GEMV family for `rows` rows and input width K
// (the staged activation tile must fit in shared memory).
int pick_rows(int rows, int K) {
    int r = gemv_rows_for(rows);
    while (r > 1 && gemv_smem_bytes(r, K) > 200 * 1024) r = (r == 16) ? 4 : 1;
    return r;
}

int decode_splits(const talker *t, int B) {
    const int want = (2 * t->n_sm + B * t->nkv - 1) / (B * t->nkv);
    return std::max(1, std::min(64, want));
}

// Attention splits of a decode step (CTAs per (row, KV group) along the cache) and whether they
// combine inside a thread-block cluster, from the longest stream's length before the step
// (captured steps are keyed by both). Measured on GB300: one or two short streams run one CTA
// per KV group up to 3 pages (no combine at all), then a cluster of 8 (one or two pages per
// split, combined on chip; 4 and 6 measured slower) up to 16 pages; longer or more streams fill the GPU in one wave,
// combined through L2, and with several streams a split walks about eight pages of the longest
// one (fewer, longer splits keep their copy pipelines busy: measured at 4, 8 and 16 streams
// against four, six and twelve pages). A single stream past 16 pages takes 16 splits, or one
// per six pages, up to one wave (B=1 at 2000 / 4096 / 8192 rows: 0.66 / 0.73 / 0.82 ms against
// 0.71 / 0.78 / 0.83 ms with a full wave of splits).
constexpr int kAttnMmMinPages = 3;

void attn_config(const talker *t, int B, int max_len, int *splits, int *cluster, int *mm) {
    const int pages_max = (max_len + 1 + kPageRows - 1) / kPageRows;
    if (B <= 2 && pages_max <= 3) {
        *splits = 1;
        *cluster = 0;
    } else if (B <= 2 && pages_max <= 2 * kAttnClusterMax) {
        *splits = kAttnClusterMax;
        *cluster = 1;
    } else {
        *cluster = 0;
        *splits = B == 1 ? std::min(decode_splits(t, B), std::max(16, (pages_max + 5) / 6))
                         : std::min(64, std::max(decode_splits(t, B), (pages_max + 7) / 8));
    }
    // the tensor-core form pays for its fragment setup from three pages per split on
    *mm = t->kv_maps_ok && (pages_max + *splits - 1) / *splits >= kAttnMmMinPages ? 1 : 0;
}

// Grow activation buffers and workspaces to cover `rows` rows with `splits`
// attention splits. Growing invalidates captured graphs (their pointers move).
talker_status ensure_capacity(talker *t, int rows, int splits) {
    const size_t need_ws = (size_t)rows * t->nq * splits * (t->hd + 4);
    const int head_grid = (t->V + kGemvWarps - 1) / kGemvWarps;
    const size_t need_head = ((size_t)rows + 16) * head_grid;   // row blocks * grid * ROWS <= (rows + 15) * grid
    const bool grow_rows = rows > t->cap_rows;
    const bool grow_ws = need_ws > t->cap_attn_ws;
    const bool grow_head = need_head > t->cap_head_part;
    if (!grow_rows && !grow_ws && !grow_head) return TALKER_OK;
    TRY_CUDA(cudaStreamSynchronize(t->st));
    drop_graphs(t);
    if (grow_rows) {
        const int cap = std::max(rows, 16);
        float **fl[] = {&t->x, &t->raw, &t->q, &t->attn, &t->act, &t->x2};
        const int widths[] = {t->H, t->qkv_n, t->qd, t->qd, t->I, t->H};
        for (int i = 0; i < 6; ++i) {
            free_ptr(*fl[i]);
            *fl[i] = nullptr;
            TRY_CUDA(cudaMalloc(fl[i], (size_t)cap * widths[i] * sizeof(float)));
        }
        // counters: QKV per (row block of up to 16 rows, head); attention per (row, kv head); head per row block
        int **il[] = {&t->qkv_cnt, &t->attn_cnt, &t->head_cnt};
        const size_t n_heads = (size_t)t->nq + 2 * t->nkv;
        const size_t counts[] = {(size_t)cap * n_heads, (size_t)cap * t->nkv, (size_t)cap};
        for (int i = 0; i < 3; ++i) {
            free_ptr(*il[i]);
            *il[i] = nullptr;
            TRY_CUDA(cudaMalloc(il[i], counts[i] * sizeof(int)));
            TRY_CUDA(cudaMemsetAsync(*il[i], 0, counts[i] * sizeof(int), t->st));
        }
        t->cap_rows = cap;
        t->cap_cnt_rows = cap;
    }
    if (grow_ws) {
        free_ptr(t->attn_ws);
        t->attn_ws = nullptr;
        TRY_CUDA(cudaMalloc(&t->attn_ws, need_ws * sizeof(float)));
        t->cap_attn_ws = need_ws;
    }
    if (grow_head) {
        free_ptr(t->head_val);
        free_ptr(t->head_idx);
        t->head_val = nullptr;
        t->head_idx = nullptr;
        TRY_CUDA(cudaMalloc(&t->head_val, need_head * sizeof(float)));
        TRY_CUDA(cudaMalloc(&t->head_idx, need_head * sizeof(int)));
        t->cap_head_part = need_head;
    }
    return TALKER_OK;
}

talker_status validate_config(const talker_config *c) {
    if (!c) return TALKER_EINVAL;
    if (c->n_layers < 1 || c->hidden < 64 || c->hidden % 64 || c->n_q_heads < 1 || c->n_kv_heads < 1) return TALKER_EINVAL;
    if (c->head_dim != 32 && c->head_dim != 64 && c->head_dim != 128) return TALKER_EINVAL;
    if (c->n_q_heads % c->n_kv_heads || c->n_q_heads / c->n_kv_heads > 8) return TALKER_EINVAL;
    if ((c->n_q_heads * c->head_dim) % 64 || c->intermediate < 64 || c->intermediate % 64) return TALKER_EINVAL;
    if (c->vocab < 8 || c->vocab % 8) return TALKER_EINVAL;
    if (!(c->rms_eps >= 0.f) || !(c->rope_theta > 0.f)) return TALKER_EINVAL;
    if ((c->weight_dtype != TALKER_DTYPE_F32 && c->weight_dtype != TALKER_DTYPE_BF16) ||
        (c->kv_dtype != TALKER_DTYPE_F32 && c->kv_dtype != TALKER_DTYPE_BF16 && c->kv_dtype != TALKER_DTYPE_Q8_0))
        return TALKER_EINVAL;
    // Q8_0 storage: bf16 weights (its prefill runs on the tensor-core path), blocks of 32 in a head
    if (c->kv_dtype == TALKER_DTYPE_Q8_0 && (c->weight_dtype != TALKER_DTYPE_BF16 || c->head_dim < 64))
        return TALKER_EINVAL;
    // the widest GEMV input must fit one staged row in shared memory
    const int kmax = std::max(std::max(c->hidden, c->n_q_heads * c->head_dim), c->intermediate);
    if (gemv_smem_bytes(1, kmax) > 200 * 1024) return TALKER_EINVAL;
    return TALKER_OK;
}

talker_status build_store(talker *t, const talker_weight_ptrs *w) {
    const int H = t->H, I = t->I;
    const size_t wsz = t->wsz;
    const size_t sz_qkv = (size_t)t->qkv_n * H * wsz, sz_o = (size_t)H * t->qd * wsz;
    const size_t sz_gu = (size_t)2 * I * H * wsz, sz_d = (size_t)H * I * wsz;
    const size_t sz_norms = (2 * (size_t)H + 2 * (size_t)t->hd) * sizeof(float);
    size_t per_layer = align_up(sz_qkv, 256) + align_up(sz_o, 256) + align_up(sz_gu, 256) + align_up(sz_d, 256) +
                       align_up(sz_norms, 256);
    size_t total = per_layer * t->c.n_layers + align_up((size_t)t->V * H * wsz, 256) + align_up(H * sizeof(float), 256);
    TRY_CUDA(cudaMalloc(&t->wstore, total));
    char *p = t->wstore;
    auto take = [&](size_t bytes) {
        char *r = p;
        p += align_up(bytes, 256);
        return r;
    };
    const cudaMemcpyKind D2D = cudaMemcpyDeviceToDevice;
    t->L.resize(t->c.n_layers);
    for (int l = 0; l < t->c.n_layers; ++l) {
        const talker_layer_ptrs &src = w->layers[l];
        const void *need[] = {src.input_norm, src.q_proj, src.k_proj, src.v_proj, src.q_norm, src.k_norm,
                              src.o_proj, src.post_norm, src.gate_proj, src.up_proj, src.down_proj};
        for (const void *n : need)
            if (!n) return TALKER_EINVAL;
        LayerDev &d = t->L[l];
        char *qkv = take(sz_qkv);
        const size_t qbytes = (size_t)t->qd * H * wsz, kbytes = (size_t)t->kvd * H * wsz;
        TRY_CUDA(cudaMemcpyAsync(qkv, src.q_proj, qbytes, D2D, t->st));
        TRY_CUDA(cudaMemcpyAsync(qkv + qbytes, src.k_proj, kbytes, D2D, t->st));
        TRY_CUDA(cudaMemcpyAsync(qkv + qbytes + kbytes, src.v_proj, kbytes, D2D, t->st));
        d.qkv = qkv;
        char *o = take(sz_o);
        TRY_CUDA(cudaMemcpyAsync(o, src.o_proj, sz_o, D2D, t->st));
        d.o = o;
        // gate row j -> row 2j, up row j -> row 2j+1 (one GEMV warp or GEMM column pair per output j)
        char *gu = take(sz_gu);
        const size_t row = (size_t)H * wsz;
        TRY_CUDA(cudaMemcpy2DAsync(gu, 2 * row, src.gate_proj, row, row, I, D2D, t->st));
        TRY_CUDA(cudaMemcpy2DAsync(gu + row, 2 * row, src.up_proj, row, row, I, D2D, t->st));
        d.gu = gu;
        char *dn = take(sz_d);
        TRY_CUDA(cudaMemcpyAsync(dn, src.down_proj, sz_d, D2D, t->st));
        d.down = dn;
        float *nrm = reinterpret_cast<float *>(take(sz_norms));
        TRY_CUDA(cudaMemcpyAsync(nrm, src.input_norm, H * sizeof(float), D2D, t->st));
        TRY_CUDA(cudaMemcpyAsync(nrm + H, src.post_norm, H * sizeof(float), D2D, t->st));
        TRY_CUDA(cudaMemcpyAsync(nrm + 2 * H, src.q_norm, t->hd * sizeof(float), D2D, t->st));
        TRY_CUDA(cudaMemcpyAsync(nrm + 2 * H + t->hd, src.k_norm, t->hd * sizeof(float), D2D, t->st));
        d.in_norm = nrm;
        d.post_norm = nrm + H;
        d.q_norm = nrm + 2 * H;
        d.k_norm = nrm + 2 * H + t->hd;
    }
    if (!w->codec_head || !w->final_norm) return TALKER_EINVAL;
    char *hw = take((size_t)t->V * H * wsz);
    TRY_CUDA(cudaMemcpyAsync(hw, w->codec_head, (size_t)t->V * H * wsz, D2D, t->st));
    t->head = hw;
    float *fn = reinterpret_cast<float *>(take(H * sizeof(float)));
    TRY_CUDA(cudaMemcpyAsync(fn, w->final_norm, H * sizeof(float), D2D, t->st));
    t->fnorm = fn;
    return TALKER_OK;
}

}  // namespace

namespace {

CacheView cache_view(const talker *t) {
    CacheView c{};
    c.maps = t->kv_maps_ok ? &t->kv_maps : nullptr;
    c.k = t->kpool;
    c.v = t->vpool;
    c.page_table = t->d_pt;
    c.pages_per_stream = t->pps;
    c.max_seq = t->max_seq;
    c.n_layers = t->c.n_layers;
    c.n_kv = t->nkv;
    c.head_dim = t->hd;
    c.kv_bf16 = t->kv_bf16;
    c.kv_q8 = t->kv_q8;
    c.page_elems = t->page_elems;
    return c;
}

struct ForwardOut {
    float *logits;
    float *hidden;
    int32_t *argmax;
    bool head_all_rows;  // logits/hidden for every row, else the last row only
    int inc_len;         // decode: bump cur_len[r] for every row after the step
    int rows_per_stream = 0;   // batched prefill: the last row of every stream (rows of T each)
    const void *head_w = nullptr;   // output head [V, H] in place of codec_head (predictor steps)
};

// The GEMV path folds the down projection into the gate/up kernel (clusters of 8 CTAs sum their
// partial products on chip) where the geometry allows: bf16 weights, I / 8 CTAs in whole
// clusters, H a multiple of 32 and at most 1024 (four down outputs per thread).
bool fuse_mlp_ok(const talker *t) {
    return t->w_bf16 && t->x2 != nullptr && t->I % 64 == 0 && t->H % 32 == 0 && t->H <= 1024;
}

// Decode attention reads the raw q|k|v projections and finishes the heads itself.
void set_raw_heads(const talker *t, const LayerDev &d, AttnParams &a) {
    a.raw = t->raw;
    a.qkv_n = t->qkv_n;
    a.q_norm = d.q_norm;
    a.k_norm = d.k_norm;
    a.rope = t->d_rope;
    a.eps = t->c.rms_eps;
}

// Enqueue the whole forward for `rows` rows on the GEMV kernels: per layer QKV (+QK-norm,
// RoPE, KV append), attention, o_proj + residual, gate/up SwiGLU, down + residual (the last
// two in one kernel where fuse_mlp_ok); then the final norm + codec_head (+argmax). Returns
// the number of kernels enqueued through *n_kernels.
talker_status enqueue_forward(talker *t, cudaStream_t st, int rows, const RowMap &rm, const float *emb,
                              int splits, const ForwardOut &out, int *n_kernels, const CodeGather *gather = nullptr) {
    const CacheView cv = cache_view(t);
    const int nh = t->c.n_layers;
    int nk = 0;
    bool pdl = false;  // the first kernel waits on everything before it in the stream
    // Fused MLP (bf16 weights): the residual stream lives in x2; o_proj writes it to x too, and
    // the gate/up kernel normalises x and reduce-adds its share of the down projection into x2.
    const bool fuse = fuse_mlp_ok(t);
    float *X = fuse ? t->x2 : t->x;
    for (int l = 0; l < nh; ++l) {
        const LayerDev &d = t->L[l];
        GemvParams p{};
        p.eps = t->c.rms_eps;
        p.rows = rows;
        p.status = t->d_status;
        // 1) RMSNorm -> [Wq;Wk;Wv] -> QK-norm, RoPE, KV append
        p.W = d.qkv;
        p.act = (l == 0) ? emb : X;
        p.act_ld = t->H;
        p.norm_w = d.in_norm;
        p.K = t->H;
        p.n_out = t->qkv_n;
        p.out = t->raw;
        p.out_ld = t->qkv_n;
        p.copy_x = (l == 0) ? X : nullptr;
        if (l == 0 && gather != nullptr) p.gather = *gather;   // rows summed from codebook tables
        p.layer = l;
        p.n_q = t->nq;
        p.n_kv = t->nkv;
        p.head_dim = t->hd;
        p.q_norm = d.q_norm;
        p.k_norm = d.k_norm;
        p.rope = t->d_rope;
        // decode rows: the attention kernel finishes the heads from the raw projections
        p.q_out = rm.mode == 0 ? nullptr : t->q;
        p.cache = cv;
        p.rowmap = rm;
        p.cnt = t->qkv_cnt;
        TRY_CUDA(launch_gemv(EPI_QKV, t->w_bf16, pick_rows(rows, t->H), p, st, pdl));
        pdl = true;
        ++nk;
        // 2) attention over [0, pos]
        AttnParams a{};
        a.q = t->q;
        a.out = t->attn;
        a.out_bf16 = 0;
        a.cache = cv;
        if (rm.mode != 0 || !t->attn_mm) a.cache.maps = nullptr;
        a.rowmap = rm;
        a.layer = l;
        a.n_q = t->nq;
        a.n_kv = t->nkv;
        a.group = t->G;
        a.splits = splits;
        a.cluster = rm.mode == 0 ? t->attn_cluster : 0;
        a.scale = 1.0f / sqrtf((float)t->hd);
        a.ws = t->attn_ws;
        a.cnt = t->attn_cnt;
        a.status = t->d_status;
        if (rm.mode == 0) set_raw_heads(t, d, a);
        TRY_CUDA(launch_attn(t->kv_kind, t->hd, a, rows, st, pdl));
        ++nk;
        // 3) o_proj + residual
        GemvParams o{};
        o.rows = rows;
        o.status = t->d_status;
        o.W = d.o;
        o.act = t->attn;
        o.act_ld = t->qd;
        o.K = t->qd;
        o.n_out = t->H;
        o.out = X;
        o.out2 = fuse ? t->x : nullptr;
        o.out_ld = t->H;
        TRY_CUDA(launch_gemv(EPI_RESID, t->w_bf16, pick_rows(rows, t->qd), o, st, pdl));
        ++nk;
        if (fuse) {
            // 4+5) post-norm -> [Wg;Wu] -> SwiGLU -> down, partials summed per cluster into x2
            GemvParams m{};
            m.rows = rows;
            m.status = t->d_status;
            m.eps = t->c.rms_eps;
            m.W = d.gu;
            m.act = t->x;
            m.act_ld = t->H;
            m.norm_w = d.post_norm;
            m.K = t->H;
            m.n_out = t->I;
            m.W2 = d.down;
            m.n_out2 = t->H;
            m.red_out = t->x2;
            TRY_CUDA(launch_gemv(EPI_SWIGLU_DOWN, t->w_bf16, pick_rows(rows, t->H), m, st, pdl));
            ++nk;
            continue;
        }
        // 4) post-norm -> [Wg;Wu] -> silu(gate) * up
        GemvParams m{};
        m.rows = rows;
        m.status = t->d_status;
        m.eps = t->c.rms_eps;
        m.W = d.gu;
        m.act = t->x;
        m.act_ld = t->H;
        m.norm_w = d.post_norm;
        m.K = t->H;
        m.n_out = t->I;
        m.out = t->act;
        m.out_ld = t->I;
        TRY_CUDA(launch_gemv(EPI_SWIGLU, t->w_bf16, pick_rows(rows, t->H), m, st, pdl));
        ++nk;
        // 5) down + residual
        GemvParams dn{};
        dn.rows = rows;
        dn.status = t->d_status;
        dn.W = d.down;
        dn.act = t->act;
        dn.act_ld = t->I;
        dn.K = t->I;
        dn.n_out = t->H;
        dn.out = t->x;
        dn.out_ld = t->H;
        TRY_CUDA(launch_gemv(EPI_RESID, t->w_bf16, pick_rows(rows, t->I), dn, st, pdl));
        ++nk;
    }
    // final norm -> codec_head -> logits, hidden, argmax
    const int hrows = out.head_all_rows ? rows : 1;
    GemvParams h{};
    h.eps = t->c.rms_eps;
    h.rows = hrows;
    h.status = t->d_status;
    h.W = out.head_w ? out.head_w : t->head;
    h.act = out.head_all_rows ? X : X + (size_t)(rows - 1) * t->H;
    h.act_ld = t->H;
    h.norm_w = t->fnorm;
    h.K = t->H;
    h.n_out = t->V;
    h.out = out.logits;
    h.out_ld = t->V;
    h.hidden_out = out.hidden;
    h.argmax_out = out.argmax;
    h.part_val = t->head_val;
    h.part_idx = t->head_idx;
    h.head_cnt = t->head_cnt;
    h.inc_len = out.inc_len;
    h.cur_len_rw = t->d_len;
    h.suppress_tail = t->suppress_tail;
    h.eos_id = t->suppress_eos;
    TRY_CUDA(launch_gemv(EPI_HEAD, t->w_bf16, pick_rows(hrows, t->H), h, st, pdl));
    ++nk;
    *n_kernels = nk;
    return TALKER_OK;
}

constexpr int kTcMinRows = 16;        // prefills shorter than this stay on the GEMV kernels
constexpr int kAttnTcMinRows = 256;   // tcgen05 prefill attention from two 128-row query tiles up (below,
                                      // its extra dense-copy launch and TMEM setup outweigh the tiles)
constexpr int kTcMinDecodeRows = 2;   // decode batches at least this wide use the tensor-core GEMMs

bool tc_usable(talker *t) {
    if (t->tc_ok < 0) {
        t->tc_ok = t->w_bf16 && gemm_tc_supported(t->qkv_n, t->H) && gemm_tc_supported(t->H, t->qd) &&
                   gemm_tc_supported(2 * t->I, t->H) && gemm_tc_supported(t->H, t->I) &&
                   prepare_gemm_tc() == cudaSuccess;
        cudaGetLastError();
    }
    return t->tc_ok == 1;
}

talker_status ensure_tc(talker *t, int rows) {
    if (rows <= t->cap_tc_rows) return TALKER_OK;
    TRY_CUDA(cudaStreamSynchronize(t->st));
    drop_graphs(t);   // captured steps hold the old buffers
    free_tc(t);
    const int cap = std::max(rows, 128);
    TRY_CUDA(cudaMalloc(&t->hb, (size_t)cap * t->H * 2));
    TRY_CUDA(cudaMalloc(&t->ab, (size_t)cap * t->qd * 2));
    TRY_CUDA(cudaMalloc(&t->gb, (size_t)cap * t->I * 2));
    TRY_CUDA(cudaMalloc(&t->gu, (size_t)cap * 2 * t->I * sizeof(float)));
    TRY_CUDA(cudaMemset(t->gu, 0, (size_t)cap * 2 * t->I * sizeof(float)));
    TRY_CUDA(cudaMalloc(&t->gemm_cnt, (size_t)(2 * t->I / 128 + 1) * sizeof(int)));
    TRY_CUDA(cudaMemset(t->gemm_cnt, 0, (size_t)(2 * t->I / 128 + 1) * sizeof(int)));
    if (t->kv_q8) TRY_CUDA(cudaMalloc(&t->kv_dense, (size_t)2 * cap * t->nkv * t->hd * 2));
    if (t->hd == 128) {   // keys of a call: up to the whole cache (an appended chunk reads every earlier key)
        const size_t lp = (size_t)attn_prefill_tc_lpad(std::max(cap, t->max_seq));
        TRY_CUDA(cudaMalloc(&t->kd_tc, lp * t->nkv * t->hd * 2));
        TRY_CUDA(cudaMalloc(&t->vt_tc, lp * t->nkv * t->hd * 2));
        t->cap_kd_keys = (int)lp;
    }
    t->cap_tc_rows = cap;
    return TALKER_OK;
}

// GEMM into `out`: reduce-added into the residual stream, or (split-K into a non-residual
// output) into zeros that an earlier kernel of the chain has written.
talker_status tc_gemm(talker *t, cudaStream_t st, const void *A, int M, int K, const void *W, int N, float *out, int ld,
                      bool residual, int *nk) {
    const int splits = gemm_tc_splits(M, N, K, t->n_sm);
    TRY_CUDA(launch_gemm_tc(A, M, K, W, N, out, ld, residual ? 1 : 0, splits, t->d_status, st));
    ++*nk;
    return TALKER_OK;
}

// Prefill of T rows at positions 0..T-1 on the tensor cores: per layer RMSNorm -> bf16,
// [Wq;Wk;Wv] GEMM, QK-norm + RoPE + KV append, causal attention, o_proj GEMM reduce-added
// into the residual stream, RMSNorm -> bf16, [Wg;Wu] GEMM, SwiGLU -> bf16, down GEMM
// reduce-added into the residual stream; then the final norm + codec_head GEMV.
talker_status enqueue_tc(talker *t, cudaStream_t st, int T, const RowMap &rm, const float *emb, int attn_splits,
                         const ForwardOut &out, int *n_kernels, const CodeGather *gather = nullptr) {
    const CacheView cv = cache_view(t);
    int nk = 0;
    // the input rows: copied in, or (gather) summed from codebook tables by layer 0's RMSNorm
    if (gather == nullptr)
        TRY_CUDA(cudaMemcpyAsync(t->x, emb, (size_t)T * t->H * sizeof(float), cudaMemcpyDeviceToDevice, st));
    for (int l = 0; l < t->c.n_layers; ++l) {
        const LayerDev &d = t->L[l];
        // a split-K QKV projection accumulates into zeros: the RMSNorm clears raw first
        const bool qkv_split = gemm_tc_splits(T, t->qkv_n, t->H, t->n_sm) > 1;
        TRY_CUDA(launch_rmsnorm_bf16(t->x, t->H, d.in_norm, t->c.rms_eps, T, t->H, t->hb, st,
                                     l == 0 ? gather : nullptr, t->d_status, qkv_split ? t->raw : nullptr,
                                     (size_t)T * t->qkv_n));
        ++nk;
        TRY(tc_gemm(t, st, t->hb, T, t->H, d.qkv, t->qkv_n, t->raw, t->qkv_n, false, &nk));
        if (rm.mode != 0) {   // prefill rows; decode rows are finished inside the attention kernel
            TRY_CUDA(launch_qkv_post(t->raw, T, t->nq, t->nkv, t->hd, d.q_norm, d.k_norm, t->d_rope, t->c.rms_eps,
                                     t->q, cv, l, rm, t->d_status, st, t->kv_q8 ? t->kv_dense : nullptr));
            ++nk;
        }
        AttnParams a{};
        a.q = t->q;
        a.out = t->ab;
        a.out_bf16 = 1;
        a.cache = cv;
        if (rm.mode != 0 || !t->attn_mm) a.cache.maps = nullptr;
        a.rowmap = rm;
        a.layer = l;
        a.n_q = t->nq;
        a.n_kv = t->nkv;
        a.group = t->G;
        a.splits = attn_splits;
        a.cluster = rm.mode == 0 ? t->attn_cluster : 0;
        a.scale = 1.0f / sqrtf((float)t->hd);
        a.ws = t->attn_ws;
        a.cnt = t->attn_cnt;
        a.status = t->d_status;
        if (rm.mode == 0) set_raw_heads(t, d, a);
        if (rm.mode == 1 && t->kv_q8) {   // the call's own rows from their dense copy, exact up to bf16
            a.dense_k = t->kv_dense;
            a.dense_v = t->kv_dense + (size_t)T * t->nkv * t->hd;
        }
        // rows of one stream: all T, or T / B in a batched prefill (B streams of rows_per_stream rows)
        const int Ts = rm.rows_per_stream > 0 ? rm.rows_per_stream : T;
        const int n_str = T / Ts;
        // (an appended chunk over Q8_0 storage attends earlier rows dequantized: tcgen05 only)
        const bool attn_tc = t->prefill_mode == 4 || (t->prefill_mode != 3 && Ts >= kAttnTcMinRows) ||
                             (t->kv_q8 && rm.pos0 > 0);
        AttnParams a1 = a;   // the first stream's rows as a one-stream call
        a1.rowmap.rows_per_stream = 0;
        if (rm.mode == 1 && attn_tc && t->kd_tc != nullptr && rm.pos0 + Ts <= t->cap_kd_keys &&
            attn_prefill_tc_supported(a1, Ts)) {
            // dense K, V^T + tcgen05 tiles, one stream after the other (the dense copy is reused)
            const size_t qrows = (size_t)Ts * t->qd, kvrows = (size_t)Ts * t->nkv * t->hd;
            for (int s = 0; s < n_str; ++s) {
                AttnParams as = a1;
                as.rowmap.stream0 = rm.stream0 + s;
                as.q = t->q + s * qrows;
                as.out = static_cast<__nv_bfloat16 *>(t->ab) + s * qrows;
                if (a.dense_k != nullptr) {
                    as.dense_k = a.dense_k + s * kvrows;
                    as.dense_v = a.dense_v + s * kvrows;
                }
                TRY_CUDA(launch_attn_prefill_tc(as, Ts, t->kd_tc, t->vt_tc, st));
                nk += 2;
            }
        } else if (rm.mode == 1 && attn_prefill_supported(t->kv_kind, t->hd)) {
            TRY_CUDA(launch_attn_prefill(t->hd, a, T, st));   // causal tiles on mma.sync
            ++nk;
        } else {
            TRY_CUDA(launch_attn(t->kv_kind, t->hd, a, T, st, false));
            ++nk;
        }
        TRY(tc_gemm(t, st, t->ab, T, t->qd, d.o, t->H, t->x, t->H, true, &nk));
        TRY_CUDA(launch_rmsnorm_bf16(t->x, t->H, d.post_norm, t->c.rms_eps, T, t->H, t->hb, st));
        ++nk;
        // gate/up + SwiGLU: in the GEMM epilogue (one K pass, or split-K finished by the last split
        // of each tile), else split-K into the zeroed gu and a SwiGLU pass that zeroes it again
        const int gu_splits = gemm_tc_splits(T, 2 * t->I, t->H, t->n_sm);
        __nv_bfloat16 *gb = static_cast<__nv_bfloat16 *>(t->gb);
        if (gu_splits == 1) {
            TRY_CUDA(launch_gemm_tc_swiglu(t->hb, T, t->H, d.gu, 2 * t->I, gb, t->I, t->d_status, st));
            ++nk;
        } else if (gemm_tc_swap_ok(T, 2 * t->I, t->H)) {
            TRY_CUDA(launch_gemm_tc_swiglu_split(t->hb, T, t->H, d.gu, 2 * t->I, t->gu, gb, t->I, t->gemm_cnt,
                                                 gu_splits, t->d_status, st));
            ++nk;
        } else {
            TRY(tc_gemm(t, st, t->hb, T, t->H, d.gu, 2 * t->I, t->gu, 2 * t->I, false, &nk));
            TRY_CUDA(launch_swiglu_bf16(t->gu, T, t->I, t->gb, st));
            ++nk;
        }
        TRY(tc_gemm(t, st, t->gb, T, t->I, d.down, t->H, t->x, t->H, true, &nk));
    }
    const int rps = out.rows_per_stream;
    const int hrows = out.head_all_rows ? T : (rps > 0 ? T / rps : 1);
    GemvParams h{};
    h.eps = t->c.rms_eps;
    h.rows = hrows;
    h.status = t->d_status;
    h.W = out.head_w ? out.head_w : t->head;
    h.act = out.head_all_rows ? t->x : t->x + (size_t)((rps > 0 ? rps : T) - 1) * t->H;
    h.act_ld = (!out.head_all_rows && rps > 0) ? rps * t->H : t->H;
    h.norm_w = t->fnorm;
    h.K = t->H;
    h.n_out = t->V;
    h.out = out.logits;
    h.out_ld = t->V;
    h.hidden_out = out.hidden;
    h.argmax_out = out.argmax;
    h.part_val = t->head_val;
    h.part_idx = t->head_idx;
    h.head_cnt = t->head_cnt;
    h.inc_len = out.inc_len;
    h.cur_len_rw = t->d_len;
    h.suppress_tail = t->suppress_tail;
    h.eos_id = t->suppress_eos;
    TRY_CUDA(launch_gemv(EPI_HEAD, t->w_bf16, pick_rows(hrows, t->H), h, st, true));
    ++nk;
    *n_kernels = nk;
    return TALKER_OK;
}

talker_status check_stream(const talker *t, int stream) {
    if (!t) return TALKER_EINVAL;
    if (t->n_streams == 0) return TALKER_ESTATE;
    if (stream < 0 || stream >= t->n_streams) return TALKER_EINVAL;
    return TALKER_OK;
}

// Run `enqueue(stream, &n_kernels)` as a CUDA graph captured once per key and replayed
// afterwards (the host then issues one launch instead of a few hundred, and the tensor maps
// of the GEMMs are encoded once, at capture). Keeps the last kMaxGraphs prefill graphs.
template <typename F>
talker_status run_graph(talker *t, const std::vector<long long> &key, F enqueue) {
    PrefillGraph *pg = nullptr;
    for (auto &g : t->pgraphs)
        if (g.key == key) pg = &g;
    if (!pg) {
        if ((int)t->pgraphs.size() >= kMaxGraphs) {
            cudaGraphExecDestroy(t->pgraphs.front().exec);
            t->pgraphs.erase(t->pgraphs.begin());
        }
        int nk = 0;
        cudaGraph_t graph = nullptr;
        TRY_CUDA(cudaStreamBeginCapture(t->cap_st, cudaStreamCaptureModeThreadLocal));
        talker_status s = enqueue(t->cap_st, &nk);
        cudaError_t e = cudaStreamEndCapture(t->cap_st, &graph);
        if (s != TALKER_OK) {
            if (graph) cudaGraphDestroy(graph);
            return s;
        }
        if (e != cudaSuccess) return from_cuda(e);
        cudaGraphExec_t exec = nullptr;
        e = cudaGraphInstantiate(&exec, graph, 0);
        cudaGraphDestroy(graph);
        if (e != cudaSuccess) return from_cuda(e);
        t->pgraphs.push_back(PrefillGraph{key, exec, nk});
        pg = &t->pgraphs.back();
    }
    TRY_CUDA(cudaGraphLaunch(pg->exec, t->st));
    t->launches += pg->n_kernels;
    return TALKER_OK;
}

// Prefill rows at positions pos0 .. pos0 + T - 1 of `stream` (pos0 = 0: talker_prefill;
// pos0 = cur_len: talker_prefill_append).
talker_status prefill_impl(talker *t, int stream, const float *emb, int T, float *hidden, float *logits,
                           int32_t *argmax, bool all_rows, bool append) {
    TRY(check_stream(t, stream));
    if (!emb || !logits || T < 1) return TALKER_EINVAL;
    if (append && t->kv_q8 && t->hd != 128) return TALKER_EINVAL;   // Q8_0 appends: the tcgen05 attention
    const int pos0 = append ? t->len[stream] : 0;
    if (T > t->max_seq - pos0) return TALKER_EOVERFLOW;
    TRY_CUDA(cudaSetDevice(t->dev));
    TRY(ensure_capacity(t, T, 1));
    RowMap rm{1, stream, pos0, t->d_len};
    ForwardOut out{logits, hidden, all_rows ? nullptr : argmax, all_rows, 0};
    if (t->kv_q8 && !tc_usable(t)) return TALKER_EINVAL;
    const bool tc = t->kv_q8 || (T >= kTcMinRows && t->prefill_mode != 2 && tc_usable(t));   // Q8_0: always tc
    if (tc) TRY(ensure_tc(t, T));
    const std::vector<long long> key = {0, tc, T, stream, pos0, all_rows, t->prefill_mode,
                                        (long long)(uintptr_t)emb, (long long)(uintptr_t)hidden,
                                        (long long)(uintptr_t)logits, (long long)(uintptr_t)out.argmax};
    TRY(run_graph(t, key, [&](cudaStream_t st, int *nk) -> talker_status {
        if (tc) TRY(enqueue_tc(t, st, T, rm, emb, 1, out, nk));
        else TRY(enqueue_forward(t, st, T, rm, emb, 1, out, nk));
        TRY_CUDA(launch_set_len(t->d_len, stream, pos0 + T, st));
        ++*nk;
        return TALKER_OK;
    }));
    t->len[stream] = pos0 + T;
    return TALKER_OK;
}

}  // namespace

extern "C" {

const char *talker_status_str(talker_status s) {
    switch (s) {
        case TALKER_OK: return "ok";
        case TALKER_EINVAL: return "invalid argument";
        case TALKER_EOVERFLOW: return "KV cache overflow";
        case TALKER_ENOMEM: return "out of device memory";
        case TALKER_ECUDA: return "CUDA error";
        case TALKER_ESTATE: return "call out of order";
        case TALKER_EDEVICE: return "device status word set";
    }
    return "unknown status";
}

talker_status talker_create(const talker_config *cfg, const talker_weight_ptrs *weights, void *cuda_stream,
                            talker_t **out) {
    if (!out) return TALKER_EINVAL;
    *out = nullptr;
    TRY(validate_config(cfg));
    if (!weights || !weights->layers) return TALKER_EINVAL;
    talker *t = new talker();
    t->c = *cfg;
    t->st = static_cast<cudaStream_t>(cuda_stream);
    t->H = cfg->hidden;
    t->nq = cfg->n_q_heads;
    t->nkv = cfg->n_kv_heads;
    t->hd = cfg->head_dim;
    t->qd = t->nq * t->hd;
    t->kvd = t->nkv * t->hd;
    t->qkv_n = t->qd + 2 * t->kvd;
    t->I = cfg->intermediate;
    t->V = cfg->vocab;
    t->G = t->nq / t->nkv;
    t->w_bf16 = cfg->weight_dtype == TALKER_DTYPE_BF16;
    t->kv_bf16 = cfg->kv_dtype == TALKER_DTYPE_BF16;
    t->kv_q8 = cfg->kv_dtype == TALKER_DTYPE_Q8_0;
    t->kv_kind = t->kv_q8 ? 2 : (t->kv_bf16 ? 1 : 0);
    t->wsz = t->w_bf16 ? 2 : 4;
    t->kvsz = t->kv_q8 ? 1 : (t->kv_bf16 ? 2 : 4);   // bytes per pool unit
    talker_status s = from_cuda(cudaGetDevice(&t->dev));
    if (s == TALKER_OK) s = from_cuda(cudaDeviceGetAttribute(&t->n_sm, cudaDevAttrMultiProcessorCount, t->dev));
    if (s == TALKER_OK) s = from_cuda(prepare_kernels());
    if (s == TALKER_OK) s = from_cuda(cudaStreamCreateWithFlags(&t->cap_st, cudaStreamNonBlocking));
    if (s == TALKER_OK) s = from_cuda(cudaMalloc(&t->d_status, sizeof(int)));
    if (s == TALKER_OK) s = from_cuda(cudaMemsetAsync(t->d_status, 0, sizeof(int), t->st));
    if (s == TALKER_OK) s = build_store(t, weights);
    if (s == TALKER_OK) s = from_cuda(cudaStreamSynchronize(t->st));
    if (s != TALKER_OK) {
        talker_destroy(t);
        return s;
    }
    *out = t;
    return TALKER_OK;
}

void talker_destroy(talker_t *t) {
    if (!t) return;
    cudaSetDevice(t->dev);
    cudaStreamSynchronize(t->st);
    drop_graphs(t);
    free_workspaces(t);
    free_cache(t);
    free_ptr(t->wstore);
    free_tc(t);
    free_ptr(t->d_status);
    free_ptr(t->d_code_tables);
    free_ptr(t->d_code_vocab);
    if (t->cap_st) cudaStreamDestroy(t->cap_st);
    delete t;
}

talker_status talker_kv_init_batched(talker_t *t, int n_streams, int max_seq_len) {
    if (!t || n_streams < 1 || max_seq_len < 1) return TALKER_EINVAL;
    TRY_CUDA(cudaSetDevice(t->dev));
    TRY_CUDA(cudaStreamSynchronize(t->st));
    drop_graphs(t);
    free_cache(t);
    const int pps = (max_seq_len + kPageRows - 1) / kPageRows;
    // pool units per page: elements, or bytes for Q8_0 tiles ([64][hd] codes + [64][hd/32] fp16 scales)
    const size_t tile_units = t->kv_q8 ? (size_t)kPageRows * t->hd + (size_t)kPageRows * (t->hd / 32) * 2
                                       : (size_t)kPageRows * t->hd;
    const size_t page_elems = (size_t)t->c.n_layers * t->nkv * tile_units;
    const size_t n_pages = (size_t)n_streams * pps;
    const size_t pool_bytes = n_pages * page_elems * t->kvsz;
    TRY_CUDA(cudaMalloc(&t->kpool, pool_bytes));
    TRY_CUDA(cudaMalloc(&t->vpool, pool_bytes));
    TRY_CUDA(cudaMemsetAsync(t->kpool, 0, pool_bytes, t->st));
    TRY_CUDA(cudaMemsetAsync(t->vpool, 0, pool_bytes, t->st));
    std::vector<int> pt(n_pages);
    for (size_t i = 0; i < n_pages; ++i) pt[i] = (int)i;  // stream s owns pages [s*pps, (s+1)*pps)
    TRY_CUDA(cudaMalloc(&t->d_pt, n_pages * sizeof(int)));
    TRY_CUDA(cudaMemcpy(t->d_pt, pt.data(), n_pages * sizeof(int), cudaMemcpyHostToDevice));
    TRY_CUDA(cudaMalloc(&t->d_len, n_streams * sizeof(int)));
    TRY_CUDA(cudaMemsetAsync(t->d_len, 0, n_streams * sizeof(int), t->st));
    // RoPE table: angle p * theta^(-2i/hd) evaluated in double on the host, stored as f32 (cos, sin)
    const int half = t->hd / 2;
    std::vector<float2> rope((size_t)max_seq_len * half);
    for (int i = 0; i < half; ++i) {
        const double inv = std::pow((double)t->c.rope_theta, -2.0 * i / t->hd);
        for (int pos = 0; pos < max_seq_len; ++pos) {
            const double ang = pos * inv;
            rope[(size_t)pos * half + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
        }
    }
    TRY_CUDA(cudaMalloc(&t->d_rope, rope.size() * sizeof(float2)));
    TRY_CUDA(cudaMemcpy(t->d_rope, rope.data(), rope.size() * sizeof(float2), cudaMemcpyHostToDevice));
    TRY_CUDA(cudaStreamSynchronize(t->st));
    // bf16 pools with head_dim 128: tensor maps over [pool rows][128] for the tensor-core decode attention
    t->kv_maps_ok = false;
    const uint64_t pool_rows = (uint64_t)n_pages * page_elems / (size_t)t->hd;
    if (t->kv_bf16 && !t->kv_q8 && t->hd == 128 && pool_rows < (1ull << 31))
        t->kv_maps_ok = make_map_bf16_2d(&t->kv_maps.k, t->kpool, pool_rows, 128, 256, 64, 64) &&
                        make_map_bf16_2d(&t->kv_maps.v, t->vpool, pool_rows, 128, 256, 64, 64);
    t->n_streams = n_streams;
    t->max_seq = max_seq_len;
    t->pps = pps;
    t->page_elems = page_elems;
    t->len.assign(n_streams, 0);
    return TALKER_OK;
}

talker_status talker_kv_rewind(talker_t *t, int stream, int new_len) {
    TRY(check_stream(t, stream));
    if (new_len < 0 || new_len > t->len[stream]) return TALKER_EINVAL;
    TRY_CUDA(cudaSetDevice(t->dev));
    TRY_CUDA(launch_set_len(t->d_len, stream, new_len, t->st));
    t->launches += 1;
    t->len[stream] = new_len;
    return TALKER_OK;
}

talker_status talker_cur_len(const talker_t *t, int stream, int *out_len) {
    TRY(check_stream(t, stream));
    if (!out_len) return TALKER_EINVAL;
    *out_len = t->len[stream];
    return TALKER_OK;
}

talker_status talker_prefill(talker_t *t, int stream, const float *emb, int T, float *hidden_last,
                             float *logits_last, int32_t *argmax_last) {
    return prefill_impl(t, stream, emb, T, hidden_last, logits_last, argmax_last, false, false);
}

talker_status talker_prefill_all_rows(talker_t *t, int stream, const float *emb, int T, float *hidden,
                                      float *logits) {
    return prefill_impl(t, stream, emb, T, hidden, logits, nullptr, true, false);
}

talker_status talker_prefill_append(talker_t *t, int stream, const float *emb, int T, float *hidden_last,
                                    float *logits_last, int32_t *argmax_last) {
    return prefill_impl(t, stream, emb, T, hidden_last, logits_last, argmax_last, false, true);
}

talker_status talker_prefill_batched(talker_t *t, int B, const float *emb, int T, float *hidden_last,
                                     float *logits_last, int32_t *argmax_last) {
    if (!t) return TALKER_EINVAL;
    if (t->n_streams == 0) return TALKER_ESTATE;
    if (!emb || !logits_last || B < 1 || B > t->n_streams || T < 1) return TALKER_EINVAL;
    if (T > t->max_seq) return TALKER_EOVERFLOW;
    if (!tc_usable(t) || (long long)B * T > (1 << 30)) return TALKER_EINVAL;   // tensor-core path only
    TRY_CUDA(cudaSetDevice(t->dev));
    const int rows = B * T;
    TRY(ensure_capacity(t, rows, 1));
    TRY(ensure_tc(t, rows));
    RowMap rm{1, 0, 0, t->d_len, T};
    ForwardOut out{logits_last, hidden_last, argmax_last, false, 0, T};
    const std::vector<long long> key = {1, B, T, t->prefill_mode, (long long)(uintptr_t)emb,
                                        (long long)(uintptr_t)hidden_last, (long long)(uintptr_t)logits_last,
                                        (long long)(uintptr_t)argmax_last};
    TRY(run_graph(t, key, [&](cudaStream_t st, int *nk) -> talker_status {
        TRY(enqueue_tc(t, st, rows, rm, emb, 1, out, nk));
        for (int s = 0; s < B; ++s) TRY_CUDA(launch_set_len(t->d_len, s, T, st));
        *nk += B;
        return TALKER_OK;
    }));
    for (int s = 0; s < B; ++s) t->len[s] = T;
    return TALKER_OK;
}

// One decode step of streams 0..B-1 as a replayed CUDA graph; the input rows come from emb, or
// (gather != null) are summed from codebook tables inside the step's first kernel.
static talker_status decode_impl(talker *t, const float *emb, const CodeGather *gather, int B, float *logits,
                                 float *hidden, int32_t *argmax) {
    if (!t) return TALKER_EINVAL;
    if (t->n_streams == 0) return TALKER_ESTATE;
    if ((!emb && !gather) || !logits || B < 1 || B > t->n_streams) return TALKER_EINVAL;
    for (int b = 0; b < B; ++b)
        if (t->len[b] + 1 > t->max_seq) return TALKER_EOVERFLOW;
    TRY_CUDA(cudaSetDevice(t->dev));
    const int kind = (t->decode_mode == 3 || (t->decode_mode == 0 && B >= kTcMinDecodeRows)) && tc_usable(t) ? 1 : 0;
    if (t->decode_mode == 3 && kind == 0) return TALKER_EINVAL;
    int max_len = 0;
    for (int b = 0; b < B; ++b) max_len = std::max(max_len, t->len[b]);
    int splits = 0, cluster = 0, mm = 0;
    attn_config(t, B, max_len, &splits, &cluster, &mm);
    TRY(ensure_capacity(t, B, splits));
    if (kind == 1) TRY(ensure_tc(t, B));
    GraphEntry *ge = nullptr;
    const int32_t *ids = gather ? gather->ids : nullptr;
    const float *overlay = gather ? gather->overlay : nullptr;
    for (auto &g : t->graphs)
        if (g.kind == kind && g.B == B && g.splits == splits && g.cluster == cluster && g.mm == mm && g.emb == emb &&
            g.logits == logits && g.hidden == hidden && g.argmax == argmax && g.ids == ids && g.overlay == overlay)
            ge = &g;
    if (!ge) {
        if ((int)t->graphs.size() >= kMaxGraphs) {
            cudaGraphExecDestroy(t->graphs.front().exec);
            t->graphs.erase(t->graphs.begin());
        }
        RowMap rm{0, 0, 0, t->d_len};
        ForwardOut out{logits, hidden, argmax, true, 1};
        int nk = 0;
        cudaGraph_t graph = nullptr;
        t->attn_cluster = cluster;
        t->attn_mm = mm;
        TRY_CUDA(cudaStreamBeginCapture(t->cap_st, cudaStreamCaptureModeThreadLocal));
        talker_status s = kind == 1 ? enqueue_tc(t, t->cap_st, B, rm, emb, splits, out, &nk, gather)
                                    : enqueue_forward(t, t->cap_st, B, rm, emb, splits, out, &nk, gather);
        cudaError_t e = cudaStreamEndCapture(t->cap_st, &graph);
        if (s != TALKER_OK) {
            if (graph) cudaGraphDestroy(graph);
            return s;
        }
        if (e != cudaSuccess) return from_cuda(e);
        cudaGraphExec_t exec = nullptr;
        e = cudaGraphInstantiate(&exec, graph, 0);
        cudaGraphDestroy(graph);
        if (e != cudaSuccess) return from_cuda(e);
        t->graphs.push_back(GraphEntry{kind, B, splits, cluster, mm, emb, logits, hidden, argmax, ids, overlay, exec, nk});
        ge = &t->graphs.back();
    }
    TRY_CUDA(cudaGraphLaunch(ge->exec, t->st));
    t->launches += ge->n_kernels;
    for (int b = 0; b < B; ++b) t->len[b] += 1;
    return TALKER_OK;
}

talker_status talker_decode(talker_t *t, const float *emb, int B, float *logits, float *hidden, int32_t *argmax) {
    return decode_impl(t, emb, nullptr, B, logits, hidden, argmax);
}

talker_status talker_kv_import(talker_t *t, int stream, const void *k, const void *v, int len) {
    TRY(check_stream(t, stream));
    if (!k || !v || len < 0) return TALKER_EINVAL;
    if (len > t->max_seq) return TALKER_EOVERFLOW;
    TRY_CUDA(cudaSetDevice(t->dev));
    TRY_CUDA(launch_kv_copy(cache_view(t), stream, const_cast<void *>(k), const_cast<void *>(v), len, 1, t->st));
    TRY_CUDA(launch_set_len(t->d_len, stream, len, t->st));
    t->launches += (len > 0) + 1;
    t->len[stream] = len;
    return TALKER_OK;
}

talker_status talker_kv_export(const talker_t *t, int stream, void *k, void *v, int len) {
    TRY(check_stream(t, stream));
    if (!k || !v || len < 0) return TALKER_EINVAL;
    if (len > t->max_seq) return TALKER_EOVERFLOW;
    TRY_CUDA(cudaSetDevice(t->dev));
    TRY_CUDA(launch_kv_copy(cache_view(t), stream, k, v, len, 0, t->st));
    const_cast<talker *>(t)->launches += (len > 0);
    return TALKER_OK;
}

talker_status talker_sync_status(talker_t *t, int32_t *code) {
    if (!t) return TALKER_EINVAL;
    TRY_CUDA(cudaSetDevice(t->dev));
    TRY_CUDA(cudaStreamSynchronize(t->st));
    int h = 0;
    TRY_CUDA(cudaMemcpy(&h, t->d_status, sizeof(int), cudaMemcpyDeviceToHost));
    if (code) *code = h;
    if (h != 0) {
        TRY_CUDA(cudaMemset(t->d_status, 0, sizeof(int)));
        return TALKER_EDEVICE;
    }
    return TALKER_OK;
}

int64_t talker_kernel_launches(const talker_t *t) { return t ? t->launches : 0; }

const char *talker_last_error(void) { return g_last_error; }

talker_status talker_test_gemm_bf16(const void *A, int M, int K, const void *B, int N, float *out, int accumulate,
                                    int splits, void *cuda_stream) {
    if (!A || !B || !out || M < 1 || splits < 1 || !gemm_tc_supported(N, K)) return TALKER_EINVAL;
    static int *d_status = nullptr;
    if (!d_status) {
        TRY_CUDA(cudaMalloc(&d_status, sizeof(int)));
        TRY_CUDA(cudaMemset(d_status, 0, sizeof(int)));
    }
    TRY_CUDA(prepare_gemm_tc());
    TRY_CUDA(launch_gemm_tc(A, M, K, B, N, out, N, accumulate, splits, d_status,
                            static_cast<cudaStream_t>(cuda_stream)));
    TRY_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream)));
    int h = 0;
    TRY_CUDA(cudaMemcpy(&h, d_status, sizeof(int), cudaMemcpyDeviceToHost));
    return h ? TALKER_EDEVICE : TALKER_OK;
}

talker_status talker_test_gemm_swiglu_bf16(const void *A, int M, int K, const void *B, int N, void *out_bf16,
                                           void *cuda_stream) {
    if (!A || !B || !out_bf16 || M < 1 || N % 2 || !gemm_tc_supported(N, K)) return TALKER_EINVAL;
    static int *d_status = nullptr;
    if (!d_status) {
        TRY_CUDA(cudaMalloc(&d_status, sizeof(int)));
        TRY_CUDA(cudaMemset(d_status, 0, sizeof(int)));
    }
    TRY_CUDA(prepare_gemm_tc());
    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
    int n_sm = 0, dev = 0;
    TRY_CUDA(cudaGetDevice(&dev));
    TRY_CUDA(cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev));
    const int splits = gemm_tc_splits(M, N, K, n_sm);
    int h = 0;
    if (splits > 1 && gemm_tc_swap_ok(M, N, K)) {
        // the runtime's split-K form: zeroed accumulator and counters, which must be zeros again after
        const size_t acc_n = (size_t)M * N, cnt_n = (size_t)N / 128;
        float *acc = nullptr;
        int *cnt = nullptr;
        TRY_CUDA(cudaMalloc(&acc, acc_n * sizeof(float)));
        TRY_CUDA(cudaMalloc(&cnt, cnt_n * sizeof(int)));
        TRY_CUDA(cudaMemsetAsync(acc, 0, acc_n * sizeof(float), st));
        TRY_CUDA(cudaMemsetAsync(cnt, 0, cnt_n * sizeof(int), st));
        TRY_CUDA(launch_gemm_tc_swiglu_split(A, M, K, B, N, acc, static_cast<__nv_bfloat16 *>(out_bf16), N / 2, cnt,
                                             splits, d_status, st));
        TRY_CUDA(cudaStreamSynchronize(st));
        std::vector<float> a(acc_n);
        std::vector<int> c(cnt_n);
        TRY_CUDA(cudaMemcpy(a.data(), acc, acc_n * sizeof(float), cudaMemcpyDeviceToHost));
        TRY_CUDA(cudaMemcpy(c.data(), cnt, cnt_n * sizeof(int), cudaMemcpyDeviceToHost));
        cudaFree(acc);
        cudaFree(cnt);
        for (float v : a) h |= v != 0.f;
        for (int v : c) h |= v != 0;
        if (h) {
            snprintf(g_last_error, sizeof(g_last_error), "split-K SwiGLU left its accumulator or counters non-zero");
            return TALKER_EDEVICE;
        }
    } else {
        TRY_CUDA(launch_gemm_tc_swiglu(A, M, K, B, N, static_cast<__nv_bfloat16 *>(out_bf16), N / 2, d_status, st));
        TRY_CUDA(cudaStreamSynchronize(st));
    }
    TRY_CUDA(cudaMemcpy(&h, d_status, sizeof(int), cudaMemcpyDeviceToHost));
    return h ? TALKER_EDEVICE : TALKER_OK;
}

talker_status talker_set_logit_suppression(talker_t *t, int vocab_tail, int eos_id) {
    if (!t || vocab_tail < 0) return TALKER_EINVAL;
    t->suppress_tail = std::min(vocab_tail, t->V);
    t->suppress_eos = eos_id;
    drop_graphs(t);   // the head's parameters are baked into captured steps
    return TALKER_OK;
}

talker_status talker_set_code_tables(talker_t *t, const void *const *tables, const int *vocab, int n_tables,
                                     int dtype) {
    if (!t || n_tables < 0 || n_tables > 32 || (n_tables > 0 && (!tables || !vocab))) return TALKER_EINVAL;
    if (dtype != TALKER_DTYPE_F32 && dtype != TALKER_DTYPE_BF16) return TALKER_EINVAL;
    for (int g = 0; g < n_tables; ++g)
        if (!tables[g] || vocab[g] < 1) return TALKER_EINVAL;
    TRY_CUDA(cudaSetDevice(t->dev));
    if (!t->d_code_tables) {
        TRY_CUDA(cudaMalloc(&t->d_code_tables, 32 * sizeof(void *)));
        TRY_CUDA(cudaMalloc(&t->d_code_vocab, 32 * sizeof(int)));
    }
    // captured steps read these device copies when they run: let queued work finish first
    TRY_CUDA(cudaStreamSynchronize(t->st));
    if (n_tables > 0) {
        TRY_CUDA(cudaMemcpy(t->d_code_tables, tables, n_tables * sizeof(void *), cudaMemcpyHostToDevice));
        TRY_CUDA(cudaMemcpy(t->d_code_vocab, vocab, n_tables * sizeof(int), cudaMemcpyHostToDevice));
    }
    t->code_tables.assign(tables, tables + n_tables);
    t->code_vocab.assign(vocab, vocab + n_tables);
    t->code_bf16 = dtype == TALKER_DTYPE_BF16;
    drop_graphs(t);   // captured steps bake the table count and type in
    return TALKER_OK;
}

talker_status talker_frame(talker_t *t, const float *emb, int T0, int n_steps, const int *table_of_step,
                           const void *const *heads, int32_t *codes, float *logits) {
    if (!t) return TALKER_EINVAL;
    const int n_tables = (int)t->code_tables.size();
    if (t->n_streams == 0 || n_tables == 0) return TALKER_ESTATE;
    if (!emb || !codes || T0 < 1 || n_steps < 0 || (n_steps > 0 && !table_of_step)) return TALKER_EINVAL;
    for (int i = 0; i < n_steps; ++i)
        if (table_of_step[i] < 0 || table_of_step[i] >= n_tables) return TALKER_EINVAL;
    if (heads)
        for (int i = 0; i <= n_steps; ++i)
            if (!heads[i]) return TALKER_EINVAL;
    auto head_of = [&](int i) -> const void * { return heads ? heads[i] : t->head; };
    if (T0 > t->max_seq || n_steps > t->max_seq - T0) return TALKER_EOVERFLOW;
    TRY_CUDA(cudaSetDevice(t->dev));
    const bool tc_pre = t->kv_q8 || (T0 >= kTcMinRows && t->prefill_mode != 2 && tc_usable(t));
    if (t->kv_q8 && !tc_usable(t)) return TALKER_EINVAL;
    // every buffer the frame touches, sized before capture (growing drops captured graphs)
    const int splits_max = std::max(kAttnClusterMax, decode_splits(t, 1));
    TRY(ensure_capacity(t, T0, splits_max));
    if (tc_pre) TRY(ensure_tc(t, T0));
    if (!t->frame_logits) {
        drop_graphs(t);
        TRY_CUDA(cudaMalloc(&t->frame_logits, (size_t)t->V * sizeof(float)));
    }
    std::vector<const void *> key = {emb, codes, logits};
    for (int i = 0; i < n_steps; ++i) key.push_back(t->code_tables[table_of_step[i]]);
    for (int i = 0; i <= n_steps; ++i) key.push_back(head_of(i));
    if (!(t->frame_exec && t->frame_T0 == T0 && t->frame_steps == n_steps && t->frame_key == key)) {
        if (t->frame_exec) cudaGraphExecDestroy(t->frame_exec);
        t->frame_exec = nullptr;
        int nk = 0;
        cudaGraph_t graph = nullptr;
        TRY_CUDA(cudaStreamBeginCapture(t->cap_st, cudaStreamCaptureModeThreadLocal));
        talker_status st = TALKER_OK;
        {   // prefill of stream 0 from position 0; code 0 = its argmax
            RowMap rm{1, 0, 0, t->d_len};
            ForwardOut out{logits ? logits : t->frame_logits, nullptr, codes, false, 0};
            out.head_w = head_of(0);
            st = tc_pre ? enqueue_tc(t, t->cap_st, T0, rm, emb, 1, out, &nk)
                        : enqueue_forward(t, t->cap_st, T0, rm, emb, 1, out, &nk);
            if (st == TALKER_OK) st = from_cuda(launch_set_len(t->d_len, 0, T0, t->cap_st));
            ++nk;
        }
        for (int i = 0; i < n_steps && st == TALKER_OK; ++i) {
            // step i: one decode step whose input row is the row of code i in its table, gathered
            // by the step's first kernel; code i + 1 = its argmax
            const int g = table_of_step[i];
            CodeGather cg{};
            cg.tables = t->d_code_tables + g;
            cg.vocab = t->d_code_vocab + g;
            cg.n = 1;
            cg.bf16 = t->code_bf16;
            cg.ids = codes + i;
            cg.ids_stride = 1;
            const int len = T0 + i;   // cache length before the step
            int splits = 0;
            attn_config(t, 1, len, &splits, &t->attn_cluster, &t->attn_mm);
            RowMap rm{0, 0, 0, t->d_len};
            ForwardOut out{logits ? logits + (size_t)(i + 1) * t->V : t->frame_logits, nullptr, codes + i + 1, false, 1};
            out.head_w = head_of(i + 1);
            if (st == TALKER_OK) st = enqueue_forward(t, t->cap_st, 1, rm, nullptr, splits, out, &nk, &cg);
        }
        cudaError_t e = cudaStreamEndCapture(t->cap_st, &graph);
        if (st != TALKER_OK) {
            if (graph) cudaGraphDestroy(graph);
            return st;
        }
        if (e != cudaSuccess) return from_cuda(e);
        e = cudaGraphInstantiate(&t->frame_exec, graph, 0);
        cudaGraphDestroy(graph);
        if (e != cudaSuccess) {
            t->frame_exec = nullptr;
            return from_cuda(e);
        }
        t->frame_T0 = T0;
        t->frame_steps = n_steps;
        t->frame_key = key;
        t->frame_kernels = nk;
    }
    TRY_CUDA(cudaGraphLaunch(t->frame_exec, t->st));
    t->launches += t->frame_kernels;
    t->len[0] = T0 + n_steps;
    return TALKER_OK;
}

talker_status talker_decode_codes(talker_t *t, const int32_t *ids, const float *overlay, int B, float *logits,
                                  float *hidden, int32_t *argmax) {
    if (!t) return TALKER_EINVAL;
    if (t->n_streams == 0 || t->code_tables.empty()) return TALKER_ESTATE;
    if (!ids) return TALKER_EINVAL;
    CodeGather cg{};
    cg.tables = t->d_code_tables;
    cg.vocab = t->d_code_vocab;
    cg.n = (int)t->code_tables.size();
    cg.bf16 = t->code_bf16;
    cg.ids = ids;
    cg.ids_stride = B;
    cg.overlay = overlay;
    return decode_impl(t, nullptr, &cg, B, logits, hidden, argmax);
}

talker_status talker_set_prefill_mode(talker_t *t, int mode) {
    if (!t || (mode != 0 && mode != 2 && mode != 3 && mode != 4)) return TALKER_EINVAL;
    t->prefill_mode = mode;
    return TALKER_OK;
}

talker_status talker_set_decode_mode(talker_t *t, int mode) {
    if (!t || (mode != 0 && mode != 2 && mode != 3)) return TALKER_EINVAL;
    t->decode_mode = mode;
    return TALKER_OK;
}

}  // extern "C"
