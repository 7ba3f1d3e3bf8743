// Region selection for sparse decode on GB300 (sm_103a).
//
// The adapter page "vllm.models.step5.nvidia.flashinfer_sparse" selects each
// decode row's regions with `select_regions(scores, current, topk,
// topk_lengths=..., sort=False)` before `sparse_decode_attention`; the body
// is not on the page.  This kernel implements the reading declared in
// include/sdattn.h: candidates are ids [0, topk_lengths[r]), the current
// region is always kept, the other topk - 1 slots take the highest scores
// (NaN lowest, ties to the lower id), and the output lists the current region
// first, then the others in ascending id order, padded with -1.
//
// One CTA per row.  A 4-pass radix select (8-bit digits) finds the key of the
// last kept score: each pass streams the row (8 loads in flight per thread;
// later passes hit L2) into per-warp shared histograms.  An ordered block scan
// over 8 consecutive ids per thread then writes the kept ids.
#include <cuda_runtime.h>

#include <cstdint>

#include "sdattn.h"

namespace {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelBatch = 8;                     // loads in flight per thread and pass

struct SelectParams {
    const float *scores;
    int64_t s_s0;
    const int32_t *current;
    int64_t cur_s0;
    const int32_t *lengths;   // NULL: every row has n_cols candidates
    int64_t len_s0;
    int32_t *out;
    int64_t out_s0;
    int rows, n_cols, topk;
};

// Order-preserving key: a larger score gives a larger key; NaN is the
// smallest key and -0 equals +0.
__device__ __forceinline__ uint32_t score_key(float x)
{
    if (x != x)
        return 0u;
    uint32_t u = __float_as_uint(x);
    if ((u & 0x7FFFFFFFu) == 0u)
        u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive block-wide prefix sum of `v` in thread order; *total gets the
// block's sum.  Uses `cnt` (kSelWarps words) and two barriers.
__device__ __forceinline__ int block_excl_sum(int v, uint32_t *cnt, int *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(~0u, incl, o);
        if (lane >= o)
            incl += x;
    }
    if (lane == 31)
        cnt[warp] = static_cast<uint32_t>(incl);
    __syncthreads();
    int before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < kSelWarps; ++w) {
        const int c = static_cast<int>(cnt[w]);
        before += w < warp ? c : 0;
        all += c;
    }
    __syncthreads();
    *total = all;
    return before + incl - v;
}

__global__ void __launch_bounds__(kSelThreads) sda_select_kernel(const __grid_constant__ SelectParams p)
{
    __shared__ uint32_t whist[kSelWarps][256];   // per-warp histograms
    __shared__ uint32_t hist[256];
    __shared__ uint32_t cnt[kSelWarps];
    __shared__ uint32_t found_digit, found_above;
    const int row = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5;
    const float *sc = p.scores + static_cast<int64_t>(row) * p.s_s0;
    int32_t *out = p.out + static_cast<int64_t>(row) * p.out_s0;
    int len = p.lengths ? p.lengths[row * p.len_s0] : p.n_cols;
    len = len < 0 ? 0 : (len > p.n_cols ? p.n_cols : len);
    const int cur = p.current[row * p.cur_s0];
    const bool forced = cur >= 0 && cur < len;
    const int k = p.topk - (forced ? 1 : 0);      // others to keep
    const int cand = len - (forced ? 1 : 0);      // others available

    // Keep every key > thr, and the first `take_eq` keys == thr in id order.
    const bool take_all = k >= cand;
    uint32_t thr = 0xFFFFFFFFu;
    int take_eq = 0;
    if (!take_all && k > 0) {
        uint32_t prefix = 0, mask = 0;
        int remaining = k;                         // rank of the last kept key among matches
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int i = tid; i < kSelWarps * 256; i += kSelThreads)
                (&whist[0][0])[i] = 0;
            __syncthreads();
            for (int base = 0; base < len; base += kSelThreads * kSelBatch) {
                float v[kSelBatch];
#pragma unroll
                for (int e = 0; e < kSelBatch; ++e) {
                    const int i = base + e * kSelThreads + tid;
                    v[e] = i < len ? sc[i] : __int_as_float(0x7FC00000);
                }
#pragma unroll
                for (int e = 0; e < kSelBatch; ++e) {
                    const int i = base + e * kSelThreads + tid;
                    const uint32_t key = score_key(v[e]);
                    if (i < len && !(forced && i == cur) && (key & mask) == prefix)
                        atomicAdd(&whist[warp][(key >> shift) & 255u], 1u);
                }
            }
            __syncthreads();
            for (int b = tid; b < 256; b += kSelThreads) {
                uint32_t sum = 0;
#pragma unroll
                for (int w = 0; w < kSelWarps; ++w)
                    sum += whist[w][b];
                hist[b] = sum;
            }
            __syncthreads();
            if (tid < 32) {
                // lane l holds bins 255 - 8l - j, j = 0..7 (descending)
                uint32_t c[8], sum = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    c[j] = hist[255 - 8 * tid - j];
                    sum += c[j];
                }
                uint32_t incl = sum;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t x = __shfl_up_sync(~0u, incl, o);
                    if (tid >= o)
                        incl += x;
                }
                const uint32_t excl = incl - sum;
                if (excl < static_cast<uint32_t>(remaining) && static_cast<uint32_t>(remaining) <= incl) {
                    uint32_t acc = excl;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (acc + c[j] >= static_cast<uint32_t>(remaining)) {
                            found_digit = 255u - 8u * tid - j;
                            found_above = acc;
                            break;
                        }
                        acc += c[j];
                    }
                }
            }
            __syncthreads();
            remaining -= static_cast<int>(found_above);
            prefix |= found_digit << shift;
            mask |= 255u << shift;
            __syncthreads();
        }
        thr = prefix;
        take_eq = remaining;
    }

    // Ordered compaction: the current region first, then the kept ids
    // ascending.  Thread t handles ids [tile + 8t, tile + 8t + 8).
    const int base = forced ? 1 : 0;
    if (forced && tid == 0)
        out[0] = cur;
    int written = 0, eq_seen = 0;
    for (int tile = 0; tile < len; tile += kSelThreads * kSelBatch) {
        const int i0 = tile + tid * kSelBatch;
        unsigned gt_bits = 0, eq_bits = 0;
#pragma unroll
        for (int e = 0; e < kSelBatch; ++e) {
            const int i = i0 + e;
            const bool valid = i < len && !(forced && i == cur);
            const uint32_t key = valid ? score_key(sc[i]) : 0u;
            if (valid && (take_all || (k > 0 && key > thr)))
                gt_bits |= 1u << e;
            if (valid && !take_all && k > 0 && key == thr)
                eq_bits |= 1u << e;
        }
        int eq_total, take_total;
        const int eq_before = block_excl_sum(__popc(eq_bits), cnt, &eq_total);
        unsigned take_bits = gt_bits;              // ties kept in id order up to take_eq
        int eq_idx = eq_seen + eq_before;
#pragma unroll
        for (int e = 0; e < kSelBatch; ++e)
            if ((eq_bits >> e) & 1u) {
                if (eq_idx < take_eq)
                    take_bits |= 1u << e;
                ++eq_idx;
            }
        int pos = base + written + block_excl_sum(__popc(take_bits), cnt, &take_total);
#pragma unroll
        for (int e = 0; e < kSelBatch; ++e)
            if ((take_bits >> e) & 1u)
                out[pos++] = i0 + e;
        written += take_total;
        eq_seen += eq_total;
    }
    for (int i = base + written + tid; i < p.topk; i += kSelThreads)
        out[i] = -1;
}

bool is_dims(const sda_tensor *t, int ndim)
{
    if (!t || t->ndim != ndim)
        return false;
    for (int i = 0; i < ndim; ++i)
        if (t->shape[i] < 0)
            return false;
    return true;
}

}  // namespace

extern "C" sda_status sparse_decode_select_regions(const sda_tensor *scores, const sda_tensor *current,
                                                   const sda_tensor *topk_lengths, int topk,
                                                   const sda_tensor *regions, void *stream)
{
    if (!is_dims(scores, 2) || !is_dims(current, 1) || !is_dims(regions, 2) || topk < 1)
        return SDA_ERR_INVALID;
    const int64_t rows = scores->shape[0], n_cols = scores->shape[1];
    if (scores->dtype != SDA_DTYPE_FP32 || (n_cols > 1 && scores->stride[1] != 1))
        return SDA_ERR_INVALID;
    if (current->dtype != SDA_DTYPE_INT32 || current->shape[0] != rows)
        return SDA_ERR_INVALID;
    if (regions->dtype != SDA_DTYPE_INT32 || regions->shape[0] != rows || regions->shape[1] != topk ||
        (topk > 1 && regions->stride[1] != 1))
        return SDA_ERR_INVALID;
    const bool has_len = topk_lengths && topk_lengths->data;
    if (has_len && (!is_dims(topk_lengths, 1) || topk_lengths->dtype != SDA_DTYPE_INT32 ||
                    topk_lengths->shape[0] != rows))
        return SDA_ERR_INVALID;
    if (rows > INT32_MAX || n_cols > INT32_MAX - kSelThreads * kSelBatch)
        return SDA_ERR_UNSUPPORTED;
    if (rows == 0)
        return SDA_OK;
    if (!scores->data || !current->data || !regions->data)
        return SDA_ERR_INVALID;
    SelectParams prm;
    prm.scores = static_cast<const float *>(scores->data);
    prm.s_s0 = scores->stride[0];
    prm.current = static_cast<const int32_t *>(current->data);
    prm.cur_s0 = current->stride[0];
    prm.lengths = has_len ? static_cast<const int32_t *>(topk_lengths->data) : nullptr;
    prm.len_s0 = has_len ? topk_lengths->stride[0] : 0;
    prm.out = static_cast<int32_t *>(const_cast<void *>(regions->data));
    prm.out_s0 = regions->stride[0];
    prm.rows = static_cast<int>(rows);
    prm.n_cols = static_cast<int>(n_cols);
    prm.topk = topk;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(rows));
    cfg.blockDim = dim3(kSelThreads);
    cfg.stream = static_cast<cudaStream_t>(stream);
    return cudaLaunchKernelEx(&cfg, sda_select_kernel, prm) == cudaSuccess ? SDA_OK : SDA_ERR_CUDA;
}
