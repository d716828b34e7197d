// Small bookkeeping kernels: per-stream length writes and dense <-> paged KV copies.
#include "common.cuh"
#include "kernels.cuh"

using namespace talker_dev;

namespace talker_k {

cudaError_t prepare_gemv();
cudaError_t prepare_attn();
cudaError_t prepare_attn_prefill();

__global__ void k_set_len(int *cur_len, int stream, int value) { cur_len[stream] = value; }

cudaError_t launch_set_len(int *cur_len, int stream, int value, cudaStream_t st) {
    k_set_len<<<1, 1, 0, st>>>(cur_len, stream, value);
    return cudaGetLastError();
}

// One CTA per (layer, kv head, position); threads over head_dim elements of
// 2 or 4 bytes. Dense layout [n_layers][n_kv][len][hd].
template <typename T>
__global__ void k_kv_copy(const CacheView c, int stream, T *dk, T *dv, int len, int to_cache) {
    const int pos = blockIdx.x;
    const int lh = blockIdx.y;               // layer * n_kv + head
    const int page = c.page_table[stream * c.pages_per_stream + pos / kPage];
    const size_t coff = (size_t)page * c.page_elems + ((size_t)lh * kPage + pos % kPage) * c.head_dim;
    const size_t doff = ((size_t)lh * len + pos) * c.head_dim;
    T *ck = static_cast<T *>(c.k) + coff;
    T *cv = static_cast<T *>(c.v) + coff;
    for (int i = threadIdx.x; i < c.head_dim; i += blockDim.x) {
        if (to_cache) {
            ck[i] = dk[doff + i];
            cv[i] = dv[doff + i];
        } else {
            dk[doff + i] = ck[i];
            dv[doff + i] = cv[i];
        }
    }
}

// Q8_0 storage: dense rows are f32. Import quantizes (warp w takes the block of dims
// 32w .. 32w + 31); export writes code * scale.
__global__ void k_kv_copy_q8(const CacheView c, int stream, float *dk, float *dv, int len, int to_cache) {
    const int pos = blockIdx.x;
    const int lh = blockIdx.y;               // layer * n_kv + head
    const int hd = c.head_dim, row = pos % kPage;
    const int page = c.page_table[stream * c.pages_per_stream + pos / kPage];
    const size_t tile = (size_t)kPage * hd + (size_t)kPage * (hd / 32) * 2;
    const size_t doff = ((size_t)lh * len + pos) * hd;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int w = warp; w < hd / 32; w += blockDim.x / 32) {
        const int i = 32 * w + lane;
        for (int kv = 0; kv < 2; ++kv) {
            unsigned char *t = static_cast<unsigned char *>(kv ? c.v : c.k) + (size_t)page * c.page_elems + lh * tile;
            float *d = (kv ? dv : dk) + doff;
            const int code_off = row * hd + 32 * w, scale_off = kPage * hd + (row * (hd / 32) + w) * 2;
            if (to_cache) {
                q8_store_block(t, code_off, scale_off, d[i], lane);
            } else {
                d[i] = (float)reinterpret_cast<const int8_t *>(t)[code_off + lane] *
                       __half2float(*reinterpret_cast<const __half *>(t + scale_off));
            }
        }
    }
}

cudaError_t launch_kv_copy(const CacheView &c, int stream, void *dense_k, void *dense_v, int len, int to_cache,
                           cudaStream_t st) {
    if (len <= 0) return cudaSuccess;
    dim3 grid(len, c.n_layers * c.n_kv, 1);
    if (c.kv_q8)
        k_kv_copy_q8<<<grid, 128, 0, st>>>(c, stream, static_cast<float *>(dense_k), static_cast<float *>(dense_v),
                                           len, to_cache);
    else if (c.kv_bf16)
        k_kv_copy<uint16_t><<<grid, 128, 0, st>>>(c, stream, static_cast<uint16_t *>(dense_k),
                                                   static_cast<uint16_t *>(dense_v), len, to_cache);
    else
        k_kv_copy<float><<<grid, 128, 0, st>>>(c, stream, static_cast<float *>(dense_k),
                                                static_cast<float *>(dense_v), len, to_cache);
    return cudaGetLastError();
}

cudaError_t prepare_kernels() {
    cudaError_t e = prepare_gemv();
    if (e != cudaSuccess) return e;
    e = prepare_attn_prefill_tc();
    if (e != cudaSuccess) return e;
    e = prepare_attn_prefill();
    if (e != cudaSuccess) return e;
    return prepare_attn();
}

}  // namespace talker_k
