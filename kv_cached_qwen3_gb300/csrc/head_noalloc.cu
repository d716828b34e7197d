// Allocation-free variant of the codec_head + argmax kernel.
//
// Some callers cannot allocate device memory: code running where a cudaMalloc
// would synchronise the device or break a memory-pool budget (a real-time audio
// thread, a host that hands the library fixed buffers only, a process whose
// allocator is owned by another framework). This entry point needs no handle
// and no allocation: the caller passes inputs and outputs, and the only scratch
// (per-CTA partial maxima and an arrival counter) lives in a file-scope device
// array of a fixed size that every GPU loading the library keeps until exit.
#include <cuda_runtime.h>

#include <atomic>

#include "common.cuh"
#include "talker.h"

using namespace talker_dev;

namespace {

constexpr int kNaRows = 64;         // most rows one call accepts
constexpr int kNaMaxBlocks = 1024;  // most CTAs one call uses (8 vocab rows each)
constexpr int kNaWarps = 8;

struct NoAllocScratch {
    float part_val[kNaMaxBlocks * kNaRows];
    int part_idx[kNaMaxBlocks * kNaRows];
    int arrivals;                   // counted up by the CTAs, put back to zero by the last one
};

// The scratch; its name in host code is a host-side stand-in, not a device address.
static __device__ __align__(256) NoAllocScratch g_na_scratch;

constexpr int kNaRowTile = 8;      // rows that share one pass over a weight row

// A NaN logit ranks as -inf in the argmax, so a row whose logits are all NaN (or all
// -inf) selects index 0, and the result never depends on the order of the CTAs.
__device__ __forceinline__ float rank_value(float x) { return isnan(x) ? -INFINITY : x; }

// logits[r][v] = hidden[r] . W[v] for v < V, argmax[r] (lowest index on ties).
// One warp per vocabulary row; the warp reads its weight row once per tile of 8
// input rows. The CTA that arrives last reduces the per-CTA partials.
template <typename WT>
__global__ void __launch_bounds__(kNaWarps * 32) k_head_argmax_noalloc(const float *hidden, int rows, int H,
                                                                        const WT *W, int V, float *logits,
                                                                        int *argmax, NoAllocScratch *sc) {
    __shared__ float bv[kNaWarps][kNaRows];
    __shared__ int bi[kNaWarps][kNaRows];
    __shared__ int last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int v = blockIdx.x * kNaWarps + warp;
    for (int r0 = 0; r0 < rows; r0 += kNaRowTile) {
        const int nr = min(kNaRowTile, rows - r0);
        float acc[kNaRowTile];
#pragma unroll
        for (int j = 0; j < kNaRowTile; ++j) acc[j] = 0.f;
        if (v < V)
            for (int k = lane; k < H; k += 32) {
                const float w = Elem<WT>::load(W, (size_t)v * H + k);
#pragma unroll
                for (int j = 0; j < kNaRowTile; ++j)
                    if (j < nr) acc[j] = fmaf(w, hidden[(size_t)(r0 + j) * H + k], acc[j]);
            }
#pragma unroll
        for (int j = 0; j < kNaRowTile; ++j) {
            const float a = warp_sum(acc[j]);
            if (lane == 0 && j < nr) {
                if (v < V) logits[(size_t)(r0 + j) * V + v] = a;
                bv[warp][r0 + j] = (v < V) ? rank_value(a) : -INFINITY;
                bi[warp][r0 + j] = v;
            }
        }
    }
    __syncthreads();
    for (int r = threadIdx.x; r < rows; r += blockDim.x) {
        float b = -INFINITY;
        int ib = 0x7fffffff;
        for (int w = 0; w < kNaWarps; ++w)
            if (bv[w][r] > b || (bv[w][r] == b && bi[w][r] < ib)) {
                b = bv[w][r];
                ib = bi[w][r];
            }
        sc->part_val[(size_t)blockIdx.x * kNaRows + r] = b;
        sc->part_idx[(size_t)blockIdx.x * kNaRows + r] = ib;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last = (atomicAdd(&sc->arrivals, 1) == (int)gridDim.x - 1);
    __syncthreads();
    if (!last) return;
    __threadfence();
    for (int r = threadIdx.x; r < rows; r += blockDim.x) {
        float b = -INFINITY;
        int ib = 0x7fffffff;
        for (int blk = 0; blk < (int)gridDim.x; ++blk) {
            const float val = __ldcg(&sc->part_val[(size_t)blk * kNaRows + r]);
            const int idx = __ldcg(&sc->part_idx[(size_t)blk * kNaRows + r]);
            if (val > b || (val == b && idx < ib)) {
                b = val;
                ib = idx;
            }
        }
        argmax[r] = ib;
    }
    if (threadIdx.x == 0) sc->arrivals = 0;   // ready for the next call
}

// Device address of the scratch, looked up once per device (with that device current).
// Two host threads making their first call at once both look it up and store the same
// value; the slots are atomics, so that is not a data race.
NoAllocScratch *scratch_for_current_device(talker_status *st) {
    static std::atomic<NoAllocScratch *> addr[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        *st = TALKER_ECUDA;
        return nullptr;
    }
    NoAllocScratch *p = addr[dev].load(std::memory_order_relaxed);
    if (p == nullptr) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_na_scratch) != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();
            *st = TALKER_ECUDA;
            return nullptr;
        }
        p = static_cast<NoAllocScratch *>(ptr);
        addr[dev].store(p, std::memory_order_relaxed);
    }
    *st = TALKER_OK;
    return p;
}

}  // namespace

extern "C" talker_status talker_head_argmax_noalloc(const float *hidden, int rows, int hidden_size, const void *W,
                                                    int vocab, int weight_dtype, float *logits, int32_t *argmax,
                                                    void *cuda_stream) {
    if (!hidden || !W || !logits || !argmax || hidden_size < 1 || vocab < 1) return TALKER_EINVAL;
    if (weight_dtype != TALKER_DTYPE_F32 && weight_dtype != TALKER_DTYPE_BF16) return TALKER_EINVAL;
    if (rows < 1 || rows > kNaRows) return TALKER_EINVAL;
    const int blocks = (vocab + kNaWarps - 1) / kNaWarps;
    if (blocks > kNaMaxBlocks) return TALKER_EINVAL;
    talker_status st = TALKER_OK;
    NoAllocScratch *sc = scratch_for_current_device(&st);
    if (!sc) return st;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    if (weight_dtype == TALKER_DTYPE_BF16)
        k_head_argmax_noalloc<__nv_bfloat16><<<blocks, kNaWarps * 32, 0, s>>>(
            hidden, rows, hidden_size, static_cast<const __nv_bfloat16 *>(W), vocab, logits, argmax, sc);
    else
        k_head_argmax_noalloc<float><<<blocks, kNaWarps * 32, 0, s>>>(hidden, rows, hidden_size,
                                                                       static_cast<const float *>(W), vocab, logits,
                                                                       argmax, sc);
    if (cudaGetLastError() != cudaSuccess) return TALKER_ECUDA;
    return TALKER_OK;
}
