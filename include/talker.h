/*
 * talker.h — C-ABI of the GB300 KV-cached Qwen3 "Talker" decoder forward.
 *
 * The operation is the KV-cached forward of a Qwen3-style causal decoder stack
 * as defined on "qwentts.cpp/src/talker-forward.h": per layer a pre-norm
 * RMSNorm, bias-free Q/K/V projections, per-head QK-RMSNorm, 1-D NEOX RoPE
 * (the multimodal axes collapsed to one position), K/V appended to a causal
 * cache, GQA scaled-dot-product attention over [0, pos], o_proj + residual,
 * a post-attention RMSNorm, a SwiGLU MLP + residual; after the last layer a
 * final RMSNorm and the codec_head projection (talker_layer_forward,
 * talker_forward_core). The entry points follow that page's statement of the
 * problem (talker_forward_prefill, talker_forward_decode, the KV cache reset)
 * and the batched cache of "transcribe.cpp/src/causal_lm/causal_lm.cpp"
 * (kv_init_batched).
 *
 * Conventions for every entry point:
 *   - All tensor pointers are CUDA DEVICE pointers on the device that was
 *     current at talker_create, unless a comment says "host".
 *   - Matrices are row-major. Linear weights are [out, in] (in contiguous),
 *     as ggml_mul_mat(W, x) reads them. Activations are [rows, features].
 *   - Work is enqueued on the stream given to talker_create and runs
 *     asynchronously; outputs are ready once that stream reaches the point
 *     after the call. Inputs must stay valid until then.
 *   - The caller owns every pointer it passes. The library owns its weight
 *     store, KV cache, workspaces and CUDA graphs, and frees them in
 *     talker_destroy.
 *   - Errors are returned as talker_status; nothing aborts or throws. All
 *     argument and capacity checks run before any work is enqueued, and a call
 *     that fails changes no state (per-stream lengths advance only on success,
 *     as cur_len does on the page).
 *   - A handle is not thread-safe: calls on one handle must be serialised.
 */
#ifndef TALKER_H
#define TALKER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct talker talker_t; /* opaque, library-owned */

typedef enum {
    TALKER_OK = 0,
    TALKER_EINVAL = 1,    /* bad argument: null pointer, size out of range, unsupported geometry */
    TALKER_EOVERFLOW = 2, /* the call would write cache rows at or past max_seq_len */
    TALKER_ENOMEM = 3,    /* a device allocation failed */
    TALKER_ECUDA = 4,     /* a CUDA runtime call failed */
    TALKER_ESTATE = 5,    /* call out of order (e.g. prefill before talker_kv_init_batched) */
    TALKER_EDEVICE = 6    /* a kernel reported an error through the device status word */
} talker_status;

/* TALKER_DTYPE_Q8_0 is a KV-cache storage type only ("qwen3-tts" talker TurboQuantQ8_0,
 * ggml Q8_0 blocks): per head row, blocks of 32 int8 codes with an fp16 scale max|x|/127.
 * A call attends the rows cached by earlier calls dequantized and its own rows exactly.
 * It needs bf16 weights and head_dim 64 or 128; talker_prefill_append with it needs
 * head_dim 128 (EINVAL otherwise). */
typedef enum { TALKER_DTYPE_F32 = 0, TALKER_DTYPE_BF16 = 1, TALKER_DTYPE_Q8_0 = 2 } talker_dtype;

/* Geometry and storage formats (names as in the rightkit-qts TtsTransformerConfig).
 * Supported: head_dim in {32, 64, 128}; n_q_heads a multiple of n_kv_heads with
 * n_q_heads / n_kv_heads <= 8; hidden, n_q_heads*head_dim and intermediate
 * multiples of 64; vocab a multiple of 8. */
typedef struct {
    int32_t n_layers;
    int32_t hidden;
    int32_t n_q_heads;
    int32_t n_kv_heads;
    int32_t head_dim;
    int32_t intermediate;
    int32_t vocab;
    float rms_eps;        /* inside the square root of every RMSNorm, QK-norm included */
    float rope_theta;     /* NEOX RoPE frequency base */
    int32_t weight_dtype; /* talker_dtype of the linear weights (norm gains are always f32) */
    int32_t kv_dtype;     /* talker_dtype of the KV cache */
} talker_config;

/* Device pointers to one layer's weights. Linear weights are [out, in] in
 * weight_dtype: q_proj [nq*hd, H], k_proj/v_proj [nkv*hd, H], o_proj [H, nq*hd],
 * gate_proj/up_proj [I, H], down_proj [H, I]. Norm gains are f32: input_norm and
 * post_norm [H], q_norm and k_norm [hd]. */
typedef struct {
    const void *input_norm, *q_proj, *k_proj, *v_proj, *q_norm, *k_norm, *o_proj;
    const void *post_norm, *gate_proj, *up_proj, *down_proj;
} talker_layer_ptrs;

typedef struct {
    const talker_layer_ptrs *layers; /* HOST array of n_layers entries */
    const void *final_norm;          /* f32 [H] */
    const void *codec_head;          /* weight_dtype [vocab, H] */
} talker_weight_ptrs;

/* Create a handle: validates the geometry, copies and repacks the weights into
 * the library's store (packed [Wq;Wk;Wv] and row-interleaved [Wg;Wu]), so the
 * caller may free its copies once the stream has passed this call.
 * cuda_stream is a cudaStream_t (NULL = the legacy default stream).
 * Errors: EINVAL (null/unsupported), ENOMEM, ECUDA. On error *out is NULL. */
talker_status talker_create(const talker_config *cfg, const talker_weight_ptrs *weights,
                            void *cuda_stream, talker_t **out);

/* Synchronises the stream and frees everything the handle owns. NULL is a no-op. */
void talker_destroy(talker_t *t);

/* Allocate (or re-allocate) the KV cache for n_streams independent streams of
 * up to max_seq_len rows each ("causal_lm.cpp", kv_init_batched). The cache is
 * bf16 or f32 (kv_dtype), laid out per stream in pages of 64 positions; each
 * page holds [layer][kv_head][64][head_dim] for K and likewise for V. Pages are
 * zeroed and every stream's length is set to 0.
 * Errors: EINVAL (n_streams < 1, max_seq_len < 1), ENOMEM, ECUDA. */
talker_status talker_kv_init_batched(talker_t *t, int n_streams, int max_seq_len);

/* Set stream's length to new_len (0 <= new_len <= current length). Rows past
 * new_len become stale and are never read again. Errors: EINVAL, ESTATE. */
talker_status talker_kv_rewind(talker_t *t, int stream, int new_len);

/* Current length of a stream (host int). Errors: EINVAL, ESTATE. */
talker_status talker_cur_len(const talker_t *t, int stream, int *out_len);

/* Prefill ("talker-forward.h", talker_forward_prefill): rewind `stream` to 0 and
 * run T rows emb [T, H] f32 at positions 0..T-1, writing their K/V at rows
 * 0..T-1; afterwards the stream's length is T.
 * Outputs for the last row only: hidden_last [H] f32 (after the final norm;
 * may be NULL), logits_last [vocab] f32 (required), argmax_last [1] int32
 * (greedy token, lowest index on ties; may be NULL).
 * Errors: EINVAL (T < 1, null emb/logits, bad stream), EOVERFLOW (T >
 * max_seq_len), ESTATE (no cache), ECUDA. */
talker_status talker_prefill(talker_t *t, int stream, const float *emb, int T,
                             float *hidden_last, float *logits_last, int32_t *argmax_last);

/* Chunked prefill ("talker-forward.h", talker_forward_core with n_past =
 * cur_len): append T rows emb [T, H] f32 to `stream` without rewinding, at
 * positions cur_len .. cur_len + T - 1; each row attends to every cached row
 * before it. Afterwards the stream's length is cur_len + T. Outputs and
 * errors as talker_prefill (EOVERFLOW when cur_len + T > max_seq_len, with
 * nothing changed). */
talker_status talker_prefill_append(talker_t *t, int stream, const float *emb, int T,
                                    float *hidden_last, float *logits_last, int32_t *argmax_last);

/* Decode ("talker-forward.h", talker_forward_decode): one row per stream for
 * streams 0..B-1. Row b of emb [B, H] f32 runs at position cur_len[b], its K/V
 * are appended at that row, it attends to [0, cur_len[b]], and afterwards
 * cur_len[b] += 1. Outputs: logits [B, vocab] f32 (required), hidden [B, H] f32
 * after the final norm (may be NULL), argmax [B] int32 (may be NULL).
 * The step runs as one replayed CUDA graph per (B, pointer set).
 * Errors: EINVAL (B < 1 or > n_streams, null pointers), EOVERFLOW (some
 * cur_len[b] + 1 > max_seq_len), ESTATE, ECUDA. */
talker_status talker_decode(talker_t *t, const float *emb, int B, float *logits, float *hidden,
                            int32_t *argmax);

/* Batched prefill ("talker-forward.h", talker_forward_prefill for streams 0..B-1
 * at once): rewind streams 0..B-1 and run T rows each; emb is [B, T, H] f32
 * (stream-major). Outputs for the last row of every stream: hidden_last [B, H]
 * (may be NULL), logits_last [B, vocab] (required), argmax_last [B] (may be
 * NULL). Runs on the tensor-core path (bf16 weights). Errors: EINVAL (B < 1 or
 * > n_streams, T < 1, null pointers, f32 weights), EOVERFLOW (T > max_seq_len),
 * ESTATE, ECUDA. */
talker_status talker_prefill_batched(talker_t *t, int B, const float *emb, int T, float *hidden_last,
                                     float *logits_last, int32_t *argmax_last);

/* TTS loop output ("qwen3-tts" talker prefill and step, codebook-0 selection):
 * before every head's argmax (prefill, append, decode), the logits of token
 * indices [vocab - vocab_tail, vocab) other than eos_id are set to -inf, in
 * the returned logits too. vocab_tail = 0 turns it off (the default). Steps
 * captured before the call are dropped and captured again. Errors: EINVAL
 * (vocab_tail < 0). */
talker_status talker_set_logit_suppression(talker_t *t, int vocab_tail, int eos_id);

/* TTS loop input ("talker-forward.h", batched forward "input_embed"): register
 * n_tables codebook embedding tables [vocab[g], hidden] (device pointers in
 * dtype TALKER_DTYPE_F32 or _BF16, table 0 = codec_embedding, then the acoustic
 * tables). The tables stay owned by the caller and must outlive their use.
 * n_tables = 0 unregisters. Synchronises the stream (captured steps read the
 * registered pointers when they run) and drops captured steps.
 * Errors: EINVAL (n_tables > 32, null table, vocab < 1), ECUDA. */
talker_status talker_set_code_tables(talker_t *t, const void *const *tables, const int *vocab, int n_tables,
                                     int dtype);

/* Decode from codebook ids: row b of the step's input is
 *   sum_g table_g[ids[g * B + b]] + overlay[b]
 * (ids: device int32 [n_tables][B], group-major; overlay: device f32 [B, hidden]
 * or NULL), summed inside the step's first kernel (the first layer's RMSNorm +
 * QKV projection reads the table rows directly), then the step as
 * talker_decode. An id outside its table sets the device status word (ST bad
 * argument) and contributes nothing. Errors: as talker_decode; ESTATE without
 * tables. */
talker_status talker_decode_codes(talker_t *t, const int32_t *ids, const float *overlay, int B, float *logits,
                                  float *hidden, int32_t *argmax);

/* Whole frame of the code-predictor loop as one CUDA graph (rightkit-qts
 * "tts_transformer.rs", predict_remaining_codebooks_kv_with_cache: a prefill,
 * then steps whose input is the previous step's code): prefill stream 0 with T0
 * rows emb [T0, H] f32 (e.g. the talker's final hidden row written on the
 * device through talker_decode's `hidden`, and a code row); code 0 = the
 * greedy token of its last row through heads[0]; then n_steps decode steps,
 * step i (generation step i + 1 on the page) reading row code_i of the
 * registered table table_of_step[i] (host int array) and producing code i + 1
 * = the greedy token of heads[i + 1]. heads is a HOST array of n_steps + 1
 * device pointers [vocab, H] in weight_dtype (the predictor's per-codebook
 * output heads), or NULL to use codec_head for every code. The codes never
 * leave the device. Outputs: codes [n_steps + 1] int32 (required), logits
 * [n_steps + 1, vocab] f32 (may be NULL). Afterwards stream 0's length is
 * T0 + n_steps. The graph is captured once and replayed while T0, n_steps,
 * the pointers, the tables and the heads stay the same. Errors: EINVAL (bad
 * sizes, table index or a NULL head), EOVERFLOW (T0 + n_steps > max_seq_len),
 * ESTATE (no cache or no code tables), ECUDA. */
talker_status talker_frame(talker_t *t, const float *emb, int T0, int n_steps, const int *table_of_step,
                           const void *const *heads, int32_t *codes, float *logits);

/* Test support: the prefill above, but writing every row's outputs:
 * hidden [T, H] (may be NULL) and logits [T, vocab] (required). */
talker_status talker_prefill_all_rows(talker_t *t, int stream, const float *emb, int T,
                                      float *hidden, float *logits);

/* Test support, modelled on the state import/export of
 * "audio.cpp/src/models/vibevoice/decoder.cpp" (TransformerKVState):
 * copy `len` rows of a stream's cache in or out. k and v are device buffers
 * [n_layers][n_kv_heads][len][head_dim] in kv_dtype (f32 for Q8_0 storage: import
 * quantizes, export writes the dequantized values). Import sets the stream's
 * length to len. Errors: EINVAL, EOVERFLOW (len > max_seq_len), ESTATE, ECUDA. */
talker_status talker_kv_import(talker_t *t, int stream, const void *k, const void *v, int len);
talker_status talker_kv_export(const talker_t *t, int stream, void *k, void *v, int len);

/* Synchronise the handle's stream and read the device status word, which a
 * kernel sets (and never traps) when it meets an impossible condition (a
 * position past the cache, a wait that gave up, a NaN logit in argmax).
 * Returns OK, EDEVICE (status word non-zero; *code gets its bits, then the
 * word is cleared) or ECUDA. code may be NULL. */
talker_status talker_sync_status(talker_t *t, int32_t *code);

/* Human-readable name of a status code (static string). */
const char *talker_status_str(talker_status s);

/* Text of the last CUDA error that made a call on this thread return ECUDA or
 * ENOMEM (static thread-local buffer; empty if none). */
const char *talker_last_error(void);

/* Choose how talker_decode runs a step: 0 = automatic (B >= 2 with bf16
 * weights: the CUDA graph of tensor-core GEMMs; otherwise the CUDA graph of
 * GEMV kernels), 2 = always the GEMV graph, 3 = always the tensor-core graph
 * (talker_decode returns EINVAL where the chosen path cannot run).
 * Errors: EINVAL (any other mode). */
talker_status talker_set_decode_mode(talker_t *t, int mode);

/* Choose how prefill runs: 0 = automatic (tensor-core GEMMs when the weights
 * are bf16, T >= 16 and every projection shape is a multiple of the GEMM tile;
 * otherwise the GEMV kernels; the causal attention of a head_dim-128 prefill with
 * at least 256 rows per stream on tcgen05 (bf16 storage from any start
 * position, Q8_0 storage from position 0), else on mma.sync),
 * 2 = always the GEMV kernels, 3 / 4 = as 0 but the attention on mma.sync /
 * on tcgen05 (where supported) at any T (comparison and test support).
 * Errors: EINVAL. */
talker_status talker_set_prefill_mode(talker_t *t, int mode);

/* Test support: the tensor-core GEMM of the prefill path on its own,
 * out[M, N] (+)= A[M, K] B[N, K]^T with bf16 A and B and f32 out (device
 * pointers; N % 128 == 0, K % 64 == 0), in the form the runtime picks for M
 * (weights as the MMA's M operand up to 128 rows, CTA pairs for 1024 rows or
 * more with N % 256 == 0, single-CTA tiles otherwise). With accumulate or
 * splits > 1 the product is added to out. Synchronises the stream. Errors:
 * EINVAL, ECUDA, EDEVICE (a wait in the kernel gave up). */
talker_status talker_test_gemm_bf16(const void *A, int M, int K, const void *B, int N, float *out, int accumulate,
                                    int splits, void *cuda_stream);

/* Test support: the prefill's gate/up GEMM with its SwiGLU epilogue ("qwentts.cpp/src/
 * talker-forward.h", talker_layer_forward MLP: silu(gate) * up). B [N, K] bf16 holds the
 * gate and up rows interleaved (row 2j = gate_j, row 2j + 1 = up_j); out_bf16 [M, N/2]
 * receives bf16(silu(A B[2j]^T) * (A B[2j+1]^T)), silu(z) = z / (1 + exp(-z)). Device
 * pointers; N % 128 == 0, K % 64 == 0, out 16-byte aligned. Where the runtime would split K
 * (at most 128 rows), the call does the same: the splits reduce into a zeroed scratch
 * accumulator and the last split of each tile writes the SwiGLU outputs; the call then checks
 * that the accumulator and the tile counters are zeros again. Synchronises the stream.
 * Errors: EINVAL, ECUDA, EDEVICE (a wait in the kernel gave up, or the scratch was left
 * non-zero). */
talker_status talker_test_gemm_swiglu_bf16(const void *A, int M, int K, const void *B, int N, void *out_bf16,
                                           void *cuda_stream);

/* Allocation-free codec_head + argmax, for callers that cannot allocate device
 * memory (a real-time audio thread where cudaMalloc would stall, a host that
 * hands the library fixed buffers only, a process whose allocator belongs to
 * another framework). The pages have no counterpart: this is a packaging of
 * the head kernel, not part of the method.
 *   logits[r][v] = hidden[r] . W[v] (f32 accumulation), argmax[r] = the index of
 *   the largest logit of row r, the lowest index on ties; 0 <= r < rows. A NaN
 *   logit ranks as -inf, so a row whose logits are all NaN (or all -inf) gets
 *   index 0; argmax is always a valid vocabulary index.
 * hidden: device f32 [rows, hidden_size]; W: device [vocab, hidden_size] in
 * weight_dtype (talker_dtype); logits: device f32 [rows, vocab]; argmax: device
 * int32 [rows]; cuda_stream: cudaStream_t (NULL = legacy stream). No handle.
 * The call allocates nothing: its scratch (per-CTA partial maxima and an
 * arrival counter) is one fixed device array in the library, held by every GPU
 * that loads the library until the process exits. Limits: rows <= 64 and
 * vocab <= 8192; larger sizes return EINVAL. The first call on a device looks
 * up the array's device address (cudaGetSymbolAddress) with that device
 * current; make that first call before any stream capture. All calls share the
 * array, so calls that may overlap on the GPU (other streams, other threads)
 * race and give wrong results: serialise them. The arrival counter is put back
 * to zero by every call. Asynchronous on cuda_stream.
 * Errors: EINVAL, ECUDA. */
talker_status talker_head_argmax_noalloc(const float *hidden, int rows, int hidden_size, const void *W, int vocab,
                                         int weight_dtype, float *logits, int32_t *argmax, void *cuda_stream);

/* Test support: count of kernel launches the library enqueued since creation
 * (a graph replay counts each of its kernels). */
int64_t talker_kernel_launches(const talker_t *t);

#ifdef __cplusplus
}
#endif

#endif /* TALKER_H */
