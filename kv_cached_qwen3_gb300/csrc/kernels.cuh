// Parameter blocks and host launchers of the Talker kernels. Included by the
// kernel translation units and by the host runtime (talker_runtime.cu).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace talker_k {

enum Epilogue : int {
    EPI_QKV = 0,     // raw q|k|v rows; the CTA that completes a head applies QK-norm, RoPE, KV append
    EPI_RESID = 1,   // out[r][f] += acc (residual stream)
    EPI_SWIGLU = 2,  // rows 2j (gate) and 2j+1 (up): out[r][j] = silu(gate) * up
    EPI_HEAD = 3,    // logits, final hidden, argmax (last CTA), decode length bump
    EPI_SWIGLU_DOWN = 4   // SwiGLU, then this CTA's share of the down projection reduce-added into red_out
};

// Where row r of a launch sits. mode 0 (decode): stream r at position cur_len[r].
// mode 1 (prefill): stream stream0 + r / rows_per_stream at position pos0 + r % rows_per_stream
// (rows_per_stream = 0: every row in stream0).
struct RowMap {
    int mode;
    int stream0;
    int pos0;
    const int *cur_len;
    int rows_per_stream;
};
__device__ __forceinline__ int rowmap_stream(const RowMap &m, int r) {
    return m.mode == 0 ? r : (m.rows_per_stream > 0 ? m.stream0 + r / m.rows_per_stream : m.stream0);
}
__device__ __forceinline__ int rowmap_pos(const RowMap &m, int r) {
    return m.mode == 0 ? m.cur_len[r] : m.pos0 + (m.rows_per_stream > 0 ? r % m.rows_per_stream : r);
}

// Tensor maps of a bf16 K and V pool with head_dim 128, viewed as [pool rows][128] (a
// (page, layer, head) tile is 64 consecutive rows): boxes of 64 rows x 64 dims, 128-byte swizzle.
struct KvMaps {
    CUtensorMap k, v;
};

// Tensor map of a bf16 matrix [rows][cols] (row stride in bytes, a multiple of 16), boxes of
// box_cols x box_rows with the 128-byte swizzle (box_cols * 2 == 128), zero fill (gemm_tc.cu).
bool make_map_bf16_2d(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t cols, uint64_t row_stride_bytes,
                      int box_cols, int box_rows);

// The paged KV cache. Page = [n_layers][n_kv][kPage][head_dim] elements; the
// position p of stream s lives in page page_table[s * pages_per_stream + p / kPage].
struct CacheView {
    const KvMaps *maps;   // host copy of the pool's tensor maps (bf16 storage, head_dim 128), else null
    void *k;
    void *v;
    const int *page_table;
    int pages_per_stream;
    int max_seq;
    int n_layers;
    int n_kv;
    int head_dim;
    int kv_bf16;        // 1: bf16 cache, 0: f32 (Q8_0 storage: kv_q8 = 1, kv_bf16 = 0)
    int kv_q8;          // 1: Q8_0 tiles ([64][hd] int8 codes + [64][hd/32] fp16 scales); page_elems in bytes
    size_t page_elems;
};

// Decode input rows gathered from codebook tables ("talker-forward.h", batched decode graph
// input: the codebook rows summed, plus an overlay row): row b = sum_g tables[g][ids[g * ids_stride
// + b]] + overlay[b]. An id outside [0, vocab[g]) sets ST_BAD_ARG and adds nothing.
struct CodeGather {
    const void *const *tables;   // device array of n table pointers, each [vocab[g], H]
    const int *vocab;            // device array of n vocabulary sizes
    int n;                       // 0: no gather (rows come from the input buffer)
    int bf16;                    // tables are bf16 (else f32)
    const int32_t *ids;          // device [n][ids_stride], group-major
    int ids_stride;
    const float *overlay;        // device [rows][H] or null
};
// Four consecutive elements [k, k + 4) of gathered row b (H % 4 == 0).
__device__ __forceinline__ float4 gather_row4(const CodeGather &c, int b, int k, int H, int *status) {
    float4 s = c.overlay ? *reinterpret_cast<const float4 *>(c.overlay + (size_t)b * H + k) : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int g = 0; g < c.n; ++g) {
        const int id = c.ids[(size_t)g * c.ids_stride + b];
        if (id < 0 || id >= c.vocab[g]) {
            if (k == 0) atomicOr(status, 1 << 3);   // ST_BAD_ARG
            continue;
        }
        const size_t i = (size_t)id * H + k;
        if (c.bf16) {
            const uint2 u = *reinterpret_cast<const uint2 *>(static_cast<const __nv_bfloat16 *>(c.tables[g]) + i);
            s.x += __uint_as_float(u.x << 16);
            s.y += __uint_as_float(u.x & 0xffff0000u);
            s.z += __uint_as_float(u.y << 16);
            s.w += __uint_as_float(u.y & 0xffff0000u);
        } else {
            const float4 v = *reinterpret_cast<const float4 *>(static_cast<const float *>(c.tables[g]) + i);
            s.x += v.x;
            s.y += v.y;
            s.z += v.z;
            s.w += v.w;
        }
    }
    return s;
}

struct GemvParams {
    const void *W;       // [rows_w, K] weight_dtype (rows_w = n_out, or 2*n_out for SWIGLU)
    const float *act;    // [rows, act_ld] f32 input activations
    int act_ld;
    const float *norm_w; // RMSNorm gain [K] for the fused prologue (QKV, SWIGLU, HEAD)
    float eps;
    int K;
    int n_out;
    int rows;
    float *out;          // epilogue destination, row stride out_ld
    int out_ld;
    float *copy_x;       // optional: CTA column 0 copies the raw input rows here (residual init)
    CodeGather gather;   // gather.n > 0: the input rows come from codebook tables, not act
    float *out2;         // EPI_RESID: optional second destination of the same sums
    const void *W2;      // EPI_SWIGLU_DOWN: down weights [n_out2][n_out] (bf16)
    float *red_out;      // EPI_SWIGLU_DOWN: [rows][n_out2], reduce-added (holds the residual)
    int n_out2;
    // EPI_QKV
    int layer, n_q, n_kv, head_dim;
    const float *q_norm, *k_norm;
    const float2 *rope;  // [max_seq][head_dim/2] (cos, sin)
    float *q_out;        // [rows, n_q*head_dim]; null: raw projections only (attention finishes the heads)
    CacheView cache;
    RowMap rowmap;
    int *cnt;            // per (row block, head) completion counters, zero between launches
    // EPI_HEAD
    float *hidden_out;   // [rows, K] final hidden (may be null)
    int *argmax_out;     // [rows] (may be null)
    float *part_val;     // per (row block, CTA, row) partial maxima
    int *part_idx;
    int *head_cnt;       // per row block counter
    int inc_len;         // decode: last CTA does cur_len[r] += 1
    int *cur_len_rw;
    int suppress_tail;   // > 0: logits of features [n_out - suppress_tail, n_out) except eos_id become -inf
    int eos_id;
    int *status;
};

struct AttnParams {
    const float *q;      // [rows, n_q*hd] after QK-norm and RoPE
    void *out;           // [rows, n_q*hd] f32, or bf16 when out_bf16
    int out_bf16;
    CacheView cache;
    RowMap rowmap;
    int layer;
    int n_q, n_kv, group;
    int splits;          // CTAs per (row, kv head) along the sequence
    float scale;         // 1/sqrt(head_dim)
    float *ws;           // partials [rows][n_q][splits][hd + 4]
    int *cnt;            // [rows][n_kv] completion counters, zero between launches
    int *status;
    // Decode rows only (row map mode 0): when raw != null, q is not read; each CTA takes
    // its heads from the raw projections [rows][qkv_n], applies QK-norm (q_norm / k_norm
    // gains, eps) and RoPE at the row's position, and split 0 appends k / v to the cache.
    const float *raw;
    int qkv_n;
    const float *q_norm, *k_norm;
    const float2 *rope;  // [max_seq][head_dim/2] (cos, sin)
    float eps;
    // 1: the splits of a (row, KV group) run as one thread-block cluster (splits <=
    // kAttnClusterMax) and combine through distributed shared memory; ws / cnt unused
    int cluster;
    // Prefill with Q8_0 storage: the call's own K / V rows, bf16 [rows][n_kv][head_dim]
    // (exact up to bf16, not read back from the quantized cache); null otherwise
    const __nv_bfloat16 *dense_k, *dense_v;
};
constexpr int kAttnClusterMax = 8;   // portable cluster size

// Tensor-core GEMM C[M, N] (+)= A[M, K] B[N, K]^T, bf16 inputs, fp32 output.
struct GemmParams {
    int M, N, K;
    float *out;
    int ld_out;
    int accumulate;   // 1: reduce-add into out (residual stream or split-K), 0: store
    int *status;
    // SwiGLU epilogue (no split-K): with B the row-interleaved [gate; up] weights, output
    // columns 2j and 2j+1 are gate_j and up_j; instead of out, write
    // swiglu_out[row, j] = bf16(silu(gate_j) * up_j) with row stride ld_swiglu.
    __nv_bfloat16 *swiglu_out;
    int ld_swiglu;
    // Split-K SwiGLU (short-product kernel only): the K splits reduce-add [gate; up] into out,
    // which holds zeros on entry; fin_cnt[tile] counts the splits that have landed, and the
    // last one writes swiglu_out from the summed tile, zeroes the tile again and resets its counter.
    int *fin_cnt;
};

constexpr int kGemvWarps = 8;
constexpr int kGemvThreads = 256;
constexpr int kAttnThreads = 256;

// Row-block heights the GEMV family is built for.
int gemv_rows_for(int rows);
size_t gemv_smem_bytes(int rows_tmpl, int K);
size_t attn_smem_bytes(int kv_bf16, int head_dim, int group);

cudaError_t launch_gemv(int epi, int w_bf16, int rows_tmpl, const GemvParams &p, cudaStream_t st, bool pdl);
// Decode / prefill-row attention over the paged cache (kv_kind 0 f32, 1 bf16, 2 Q8_0). Decode rows
// that finish their heads from the raw projections on a bf16 or Q8_0 cache (head_dim 64 or 128,
// GQA group of 1 or 2) run the key-parallel kernel (attn_decode_keys.cu), every other case the
// split kernel.
cudaError_t launch_attn(int kv_kind, int head_dim, const AttnParams &p, int rows, cudaStream_t st, bool pdl);
bool attn_dec_keys_supported(int kv_kind, int head_dim, const AttnParams &p);
cudaError_t launch_attn_dec_keys(int kv_kind, int head_dim, const AttnParams &p, int rows, cudaStream_t st, bool pdl);
cudaError_t prepare_attn_dec_keys();
cudaError_t launch_set_len(int *cur_len, int stream, int value, cudaStream_t st);
// Copy len rows of a stream between a dense [n_layers][n_kv][len][hd] buffer and the cache.
cudaError_t launch_kv_copy(const CacheView &c, int stream, void *dense_k, void *dense_v, int len, int to_cache,
                           cudaStream_t st);
// Causal prefill attention on the tensor cores (bf16 cache, head_dim 64 or 128, row map
// mode 1, bf16 output).
bool attn_prefill_supported(int kv_bf16, int head_dim);
cudaError_t launch_attn_prefill(int head_dim, const AttnParams &a, int T, cudaStream_t st);
cudaError_t prepare_kernels();  // raise dynamic shared-memory limits once per process

// tcgen05 causal prefill attention (head_dim 128, one stream from position 0): dense K and
// V^T copies (kd, vt: n_kv * attn_prefill_tc_lpad(T) * 128 bf16 each), then the tiles.
bool attn_prefill_tc_supported(const AttnParams &a, int T);
int attn_prefill_tc_lpad(int nkeys);
cudaError_t prepare_attn_prefill_tc();
cudaError_t launch_attn_prefill_tc(const AttnParams &a, int T, __nv_bfloat16 *kd, __nv_bfloat16 *vt, cudaStream_t st);

bool gemm_tc_supported(int N, int K);
int gemm_tc_splits(int M, int N, int K, int n_sm);
cudaError_t prepare_gemm_tc();
// Short products (M <= 128) with the weights as the MMA's M operand (k_gemm_tc_swap): X bf16
// [M, K], W bf16 [N, K] (N % 128 == 0); out f32 [M, ld_out], reduce-added when accumulate or
// splits > 1 (then out must hold zeros or the residual stream); or, with swiglu_out and one
// split, bf16(silu(gate) * up) of interleaved weight rows into swiglu_out [M, N/2].
bool gemm_tc_swap_ok(int M, int N, int K);
int gemm_tc_swap_splits(int M, int N, int K, int n_sm);
cudaError_t launch_gemm_tc_swap(const void *X, int M, int K, const void *W, int N, float *out, int ld_out,
                                int accumulate, int splits, __nv_bfloat16 *swiglu_out, int ld_swiglu, int *status,
                                cudaStream_t st, int *fin_cnt = nullptr);
// Split-K gate/up with SwiGLU for M <= 128: acc f32 [M, N] must hold zeros and cnt [N / 128]
// zeros on entry, and both hold zeros again when the kernel has finished; out_bf16 [M, N/2]
// (row stride ld) receives bf16(silu(gate) * up).
cudaError_t launch_gemm_tc_swiglu_split(const void *A, int M, int K, const void *B, int N, float *acc,
                                        __nv_bfloat16 *out_bf16, int ld, int *cnt, int splits, int *status,
                                        cudaStream_t st);
// A: bf16 [M, K], B: bf16 [N, K] (device); out: f32 [M, ld_out]. With splits > 1 the
// result is reduce-added, so out must hold zeros (or the residual stream).
cudaError_t launch_gemm_tc(const void *A, int M, int K, const void *B, int N, float *out, int ld_out, int accumulate,
                           int splits, int *status, cudaStream_t st);
// The same GEMM with the SwiGLU epilogue: out_bf16 [M, N/2] (row stride ld), one K pass.
cudaError_t launch_gemm_tc_swiglu(const void *A, int M, int K, const void *B, int N, __nv_bfloat16 *out_bf16, int ld,
                                  int *status, cudaStream_t st);

// Element-wise stages of the tensor-core prefill path (prefill.cu).
// With gather.n > 0 the rows are first gathered from codebook tables and also written to x.
// With zero != null the kernel also clears zero[0 .. zero_n) (zero_n % 4 == 0, 16-byte aligned):
// the split-K accumulator of the GEMM that follows.
cudaError_t launch_rmsnorm_bf16(float *x, int ld, const float *w, float eps, int rows, int H, void *out,
                                cudaStream_t st, const CodeGather *gather = nullptr, int *status = nullptr,
                                float *zero = nullptr, size_t zero_n = 0);
// dense_kv (Q8_0 storage only, else null): the rows' k / v also go to bf16 [2][rows][n_kv][hd]
cudaError_t launch_qkv_post(const float *raw, int rows, int n_q, int n_kv, int hd, const float *q_norm,
                            const float *k_norm, const float2 *rope, float eps, float *q_out, const CacheView &cache,
                            int layer, const RowMap &rm, int *status, cudaStream_t st,
                            __nv_bfloat16 *dense_kv = nullptr);
// silu(gate) * up of a split-K [gate; up] sum; gu is zeroed behind the read (its split-K
// accumulation always starts from zeros).
cudaError_t launch_swiglu_bf16(float *gu, int rows, int I, void *out, cudaStream_t st);

}  // namespace talker_k
