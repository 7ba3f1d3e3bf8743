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
// One CTA of 256 threads per row (4 per SM), scores compared as
// order-preserving 32-bit keys; the row is prefetched into L2 at entry.
//   Fast path (rows of up to 64K candidates): a 16-bit lower bound is read
//   off a 2048-score sample so that the topk best scores pass it with a
//   margin of five binomial standard deviations; one streaming pass (a plain
//   float comparison against the bound's smallest passing value, one warp
//   ballot per 32 ids) writes a bitmap of the passing ids; their keys are
//   gathered (L2 hits) into a shared buffer in ascending id order while a
//   histogram of their 16-bit prefixes is built; the prefix holding rank topk
//   and a one-warp ranking of its few keys give the exact last kept key; one
//   block scan over the buffer places the kept ids and the lowest-id ties.
//   Fallback (buffer overflow or underflow, longer rows): an exact 4-pass
//   radix select that streams the row each pass, then an ordered compaction.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "sdattn.h"

namespace {

constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelBatch = 8;                     // loads in flight per thread (exact passes)
constexpr int kFilterBatch = 16;                 // loads in flight per thread (filter pass)
constexpr int kFilterStep = kSelThreads * kFilterBatch;
constexpr int kGather = 8;                      // candidate key loads in flight per thread
constexpr int kSample = 2048;                    // scores sampled for the filter threshold
constexpr int kBufCap = 4080;                    // candidate (key, id) pairs held in shared memory
constexpr int kFastMaxLen = 65536;               // longest row the bitmaps cover
constexpr int kBitWords = kFastMaxLen / 32;

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

struct SelShared {
    uint32_t whist[kSelWarps][256];              // per-warp histograms; row 0 then holds the sums
    uint32_t cnt[kSelWarps];
    uint32_t found[3];                           // digit (or prefix), keys above it, keys in it
    uint32_t counter;                            // fill of bin_keys
    union {
        uint32_t sample[kSample];
        struct {
            uint32_t kept[kBitWords];            // candidate bitmap of the streaming pass
            uint32_t bin_keys[32];               // keys sharing the 16-bit prefix of rank topk
        } bits;
    } a;
    uint32_t buf_key[kBufCap];
    int32_t buf_id[kBufCap];
};
// 4 CTAs per SM: 228 KB of shared memory per SM, 1 KB of it reserved per CTA.
static_assert(sizeof(SelShared) <= 4 * 1024 * 14, "selection shared memory above 4 CTAs per SM");
// The streaming pass stores one bitmap word per lane below kFilterBatch and
// never past the bitmap; the prefix histogram is the 2048 words of whist, 8
// bins per thread; the sample is 8 scores per thread.
static_assert(kFilterBatch <= 32 && kFastMaxLen % kFilterStep == 0, "streaming pass layout");
static_assert(kSelWarps * 256 == 2048 && 8 * kSelThreads == 2048, "prefix histogram layout");
static_assert(kSample % kSelThreads == 0, "sample layout");

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

// The smallest float whose key is at least t > 0: a non-NaN x has
// score_key(x) >= t exactly when x >= this value (NaN, which fails every
// ordered comparison, when no float reaches t; -inf when every float does).
__device__ __forceinline__ float key_floor_value(uint32_t t)
{
    if (t & 0x80000000u) {                               // +0 and the positive floats
        const uint32_t u = t & 0x7FFFFFFFu;
        return __uint_as_float(u > 0x7F800000u ? 0x7FC00000u : u);
    }
    const uint32_t u = ~t;                               // the negative floats
    return (u & 0x7FFFFFFFu) > 0x7F800000u ? __uint_as_float(0xFF800000u) : __uint_as_float(u);
}

// Starts pulling bytes [p, p + n) of global memory into L2 (no data is
// returned): one bulk prefetch of the 16-byte-aligned interior.
__device__ __forceinline__ void prefetch_l2(const void *p, size_t n)
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uintptr_t lo = (a + 15) & ~static_cast<uintptr_t>(15);
    const uintptr_t hi = (a + n) & ~static_cast<uintptr_t>(15);
    if (hi > lo)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(lo), "r"(static_cast<uint32_t>(hi - lo))
                     : "memory");
}

// Exclusive block-wide prefix sum of `v` in thread order; *total gets the
// block's sum.  Two barriers.
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

__device__ __forceinline__ void zero_whist(SelShared &sh)
{
    for (int i = threadIdx.x; i < kSelWarps * 256; i += kSelThreads)
        (&sh.whist[0][0])[i] = 0;
}

// Sums the per-warp histograms (into whist[0]: each bin is summed by one
// thread) and finds the digit holding the key of descending rank
// `remaining`: sh.found = {digit, keys in higher digits}.
__device__ __forceinline__ void find_digit(SelShared &sh, int remaining)
{
    const int tid = threadIdx.x;
    __syncthreads();
    for (int b = tid; b < 256; b += kSelThreads) {
        uint32_t sum = 0;
#pragma unroll
        for (int w = 0; w < kSelWarps; ++w)
            sum += sh.whist[w][b];
        sh.whist[0][b] = sum;
    }
    __syncthreads();
    if (tid < 32) {
        uint32_t c[8], sum = 0;   // lane l: bins 255 - 8l - j, j = 0..7 (descending)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            c[j] = sh.whist[0][255 - 8 * tid - j];
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
                    sh.found[0] = 255u - 8u * tid - j;
                    sh.found[1] = acc;
                    break;
                }
                acc += c[j];
            }
        }
    }
    __syncthreads();
}

// Key of descending rank `rank` (1 <= rank <= n) among keys[0, n) in shared
// memory; *above gets the number of keys strictly greater.  With `digits` < 4
// only the top 8 * digits bits are resolved and the lower bits are zero: a
// lower bound of that key.  With `first_ready` the caller has already built
// the per-warp histograms of the top digit (key >> 24) over all n keys.
__device__ uint32_t select_shared(SelShared &sh, const uint32_t *keys, int n, int rank, int *above,
                                  int digits = 4, bool first_ready = false)
{
    const int warp = threadIdx.x >> 5;
    uint32_t prefix = 0, mask = 0;
    int remaining = rank;
    for (int shift = 24; shift >= 32 - 8 * digits; shift -= 8) {
        if (!(first_ready && shift == 24)) {
            zero_whist(sh);
            __syncthreads();
            for (int i = threadIdx.x; i < n; i += kSelThreads) {
                const uint32_t key = keys[i];
                if ((key & mask) == prefix)
                    atomicAdd(&sh.whist[warp][(key >> shift) & 255u], 1u);
            }
        }
        find_digit(sh, remaining);
        remaining -= static_cast<int>(sh.found[1]);
        prefix |= sh.found[0] << shift;
        mask |= 255u << shift;
        __syncthreads();
    }
    *above = rank - remaining;
    return prefix;
}

// The same over the row's candidates in global memory (all ids < len except cur).
__device__ uint32_t select_global(SelShared &sh, const float *sc, int len, int cur, bool forced, int rank,
                                  int *above)
{
    const int tid = threadIdx.x, warp = tid >> 5;
    uint32_t prefix = 0, mask = 0;
    int remaining = rank;
    for (int shift = 24; shift >= 0; shift -= 8) {
        zero_whist(sh);
        __syncthreads();
        for (int base = 0; base < len; base += kSelThreads * kSelBatch) {
            float v[kSelBatch];
#pragma unroll
            for (int e = 0; e < kSelBatch; ++e) {
                const int i = base + e * kSelThreads + tid;
                v[e] = i < len ? sc[i] : 0.0f;
            }
#pragma unroll
            for (int e = 0; e < kSelBatch; ++e) {
                const int i = base + e * kSelThreads + tid;
                const uint32_t key = score_key(v[e]);
                if (i < len && !(forced && i == cur) && (key & mask) == prefix)
                    atomicAdd(&sh.whist[warp][(key >> shift) & 255u], 1u);
            }
        }
        find_digit(sh, remaining);
        remaining -= static_cast<int>(sh.found[1]);
        prefix |= sh.found[0] << shift;
        mask |= 255u << shift;
        __syncthreads();
    }
    *above = rank - remaining;
    return prefix;
}

__global__ void __launch_bounds__(kSelThreads, 4) sda_select_kernel(const __grid_constant__ SelectParams p)
{
    extern __shared__ __align__(16) unsigned char sel_smem[];
    SelShared &sh = *reinterpret_cast<SelShared *>(sel_smem);
    const int row = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31;
    const float *sc = p.scores + static_cast<int64_t>(row) * p.s_s0;
    int32_t *out = p.out + static_cast<int64_t>(row) * p.out_s0;
    int len = p.lengths ? p.lengths[row * p.len_s0] : p.n_cols;
    len = len < 0 ? 0 : (len > p.n_cols ? p.n_cols : len);
    const int cur = p.current[row * p.cur_s0];
    const bool forced = cur >= 0 && cur < len;
    const int k = p.topk - (forced ? 1 : 0);      // others to keep
    const int cand = len - (forced ? 1 : 0);      // others available
    const int base = forced ? 1 : 0;
    if (tid == 0) {
        if (len > 0)
            prefetch_l2(sc, static_cast<size_t>(len) * sizeof(float));
        if (forced)
            out[0] = cur;
    }

    // Keep every key > thr and the first take_eq keys == thr in id order;
    // take_all keeps every candidate, k <= 0 keeps none.
    const bool take_all = k >= cand;
    uint32_t thr = 0xFFFFFFFFu;
    int take_eq = 0;
    int written = 0;
    bool done = take_all || k <= 0;

    if (!done && len <= kFastMaxLen) {
        // ---- filter threshold from a sample (all candidates when few)
        uint32_t t_lo = 0u;
        if (cand > kBufCap) {
            // the first radix digit's histogram is built as the sample loads
            zero_whist(sh);
            __syncthreads();
            for (int j = tid; j < kSample; j += kSelThreads) {
                const uint32_t key = score_key(sc[static_cast<int64_t>(j) * len / kSample]);
                sh.a.sample[j] = key;
                atomicAdd(&sh.whist[tid >> 5][key >> 24], 1u);
            }
            // Sample rank of the bound: the sample's expected count of the row's
            // top k (a binomial mean mu) plus five standard deviations and a
            // constant, so that fewer than k candidates reach the bound only
            // with probability ~1e-7 (the exact fallback then takes the row).
            const float mu = static_cast<float>(k) * kSample / static_cast<float>(cand);
            const int r = min(kSample, static_cast<int>(mu + 5.0f * sqrtf(mu)) + 17);
            int unused;
            t_lo = select_shared(sh, sh.a.sample, kSample, r, &unused, 2, true);   // 16-bit lower bound
        }
        // ---- one streaming pass: a bitmap of the candidates with key >= t_lo.
        // Element e of a batch is id b0 + 256 e + tid, so for each e a warp's
        // lanes hold 32 consecutive ids: one ballot forms that bitmap word, and
        // lane e stores it.  With t_lo > 0 the test key >= t_lo is the float
        // comparison x >= key_floor_value(t_lo); batches wholly inside the row
        // and clear of the current region skip the per-score id checks.
        const int excl = forced ? cur : -1;
        const bool keep_all = t_lo == 0u;
        const float x_lo = keep_all ? 0.0f : key_floor_value(t_lo);
        const int warp = tid >> 5;
        for (int b0 = 0; b0 < len; b0 += kFilterStep) {
            const bool plain = !keep_all && b0 + kFilterStep <= len && (excl < b0 || excl >= b0 + kFilterStep);
            float v[kFilterBatch];
            uint32_t mine = 0;
            if (plain) {
                const float *src = sc + b0 + tid;
#pragma unroll
                for (int e = 0; e < kFilterBatch; ++e)
                    v[e] = src[e * kSelThreads];
#pragma unroll
                for (int e = 0; e < kFilterBatch; ++e) {
                    const uint32_t w = __ballot_sync(~0u, v[e] >= x_lo);
                    mine = lane == e ? w : mine;
                }
            } else {
#pragma unroll
                for (int e = 0; e < kFilterBatch; ++e) {
                    const int i = b0 + e * kSelThreads + tid;
                    v[e] = i < len ? sc[i] : 0.0f;
                }
#pragma unroll
                for (int e = 0; e < kFilterBatch; ++e) {
                    const int i = b0 + e * kSelThreads + tid;
                    const uint32_t w = __ballot_sync(~0u, i < len && i != excl && (keep_all || v[e] >= x_lo));
                    mine = lane == e ? w : mine;
                }
            }
            if (lane < kFilterBatch)   // word of ids b0 + 256 lane + 32 warp + [0, 32)
                sh.a.bits.kept[(b0 >> 5) + lane * kSelWarps + warp] = mine;
        }
        __syncthreads();
        // ---- the candidates' ids into the buffer, ascending: thread t owns
        // bitmap words [t W, t W + W)
        const int words = (len + 31) / 32;
        const int W = (words + kSelThreads - 1) / kSelThreads;
        const int w0 = tid * W, w1 = min(words, w0 + W);
        int total;
        {
            int c = 0;
            for (int w = w0; w < w1; ++w)
                c += __popc(sh.a.bits.kept[w]);
            int at = block_excl_sum(c, sh.cnt, &total);
            if (total <= kBufCap && total >= k) {
                for (int w = w0; w < w1; ++w) {   // candidate ids, ascending
                    uint32_t b = sh.a.bits.kept[w];
                    while (b) {
                        const int bit = __ffs(b) - 1;
                        b &= b - 1;
                        sh.buf_id[at++] = w * 32 + bit;
                    }
                }
            }
        }
        uint32_t *const hist = &sh.whist[0][0];   // 2048 bins: 16-bit key prefixes above t_lo's
        const uint32_t hi0 = t_lo >> 16;
        if (total <= kBufCap && total >= k) {
            if (t_lo != 0u)
                for (int b = tid; b < kSelWarps * 256; b += kSelThreads)
                    hist[b] = 0;
            if (tid == 0)
                sh.counter = 0;
            __syncthreads();
            // their keys (the row has just streamed through, so these loads hit L2)
            // and, over a 16-bit bound, the histogram of their prefixes
            for (int i0 = 0; i0 < total; i0 += kSelThreads * kGather) {
                float g[kGather];
#pragma unroll
                for (int e = 0; e < kGather; ++e) {
                    const int i = i0 + e * kSelThreads + tid;
                    g[e] = i < total ? sc[sh.buf_id[i]] : 0.0f;
                }
#pragma unroll
                for (int e = 0; e < kGather; ++e) {
                    const int i = i0 + e * kSelThreads + tid;
                    if (i < total) {
                        const uint32_t key = score_key(g[e]);
                        sh.buf_key[i] = key;
                        if (t_lo != 0u)
                            atomicAdd(&hist[min((key >> 16) - hi0, 2047u)], 1u);
                    }
                }
            }
            // ---- exact select inside the buffer: the key of descending rank k
            int above = 0;
            bool found = false;
            if (t_lo != 0u) {
                // the prefix holding rank k: thread t owns prefixes [8 (255 - t), 8 (255 - t) + 8)
                __syncthreads();
                const int hb = 8 * (kSelThreads - 1 - tid);
                uint32_t hc[8];
                int s8 = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    hc[j] = hist[hb + 7 - j];
                    s8 += static_cast<int>(hc[j]);
                }
                int all;
                const int before = block_excl_sum(s8, sh.cnt, &all);
                if (before < k && k <= before + s8) {
                    int acc = before;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (acc + static_cast<int>(hc[j]) >= k) {
                            sh.found[0] = static_cast<uint32_t>(hb + 7 - j);
                            sh.found[1] = static_cast<uint32_t>(acc);
                            sh.found[2] = hc[j];
                            break;
                        }
                        acc += static_cast<int>(hc[j]);
                    }
                }
                __syncthreads();
                // read from the finder's broadcast, not from hist, which the
                // fallback below zeroes at once: the branch is block-uniform
                const uint32_t bin = sh.found[0];
                const int above_bin = static_cast<int>(sh.found[1]);
                const int in_bin = static_cast<int>(sh.found[2]);
                if (bin < 2047u && in_bin <= 32) {
                    // the prefix's keys (at most 32) ranked by one warp
                    for (int e = tid; e < total; e += kSelThreads) {
                        const uint32_t key = sh.buf_key[e];
                        if ((key >> 16) - hi0 == bin)
                            sh.a.bits.bin_keys[atomicAdd(&sh.counter, 1u)] = key;
                    }
                    __syncthreads();
                    if (tid < 32) {
                        const uint32_t mine = tid < in_bin ? sh.a.bits.bin_keys[tid] : 0u;
                        int gt = 0, eq = 0;
                        for (int j = 0; j < in_bin; ++j) {
                            const uint32_t o = __shfl_sync(~0u, mine, j);
                            gt += o > mine;
                            eq += o == mine;
                        }
                        const int need = k - above_bin;
                        if (tid < in_bin && gt < need && need <= gt + eq) {   // equal keys write equal values
                            sh.found[0] = mine;
                            sh.found[1] = static_cast<uint32_t>(above_bin + gt);
                        }
                    }
                    __syncthreads();
                    thr = sh.found[0];
                    above = static_cast<int>(sh.found[1]);
                    found = true;
                }
            }
            if (!found)
                thr = select_shared(sh, sh.buf_key, total, k, &above);
            take_eq = k - above;
            // ---- output: the buffer's ids ascend, so thread t's slice [t C, t C + C)
            // keeps its keys above thr and its ties while fewer than take_eq precede them
            const int C = (total + kSelThreads - 1) / kSelThreads;
            const int e0 = min(total, tid * C), e1 = min(total, e0 + C);
            int strict = 0, ties = 0;
            for (int e = e0; e < e1; ++e) {
                const uint32_t key = sh.buf_key[e];
                strict += key > thr;
                ties += key == thr;
            }
            int sums;
            const int before = block_excl_sum((ties << 16) | strict, sh.cnt, &sums);
            int tie_rank = before >> 16;
            int pos = base + (before & 0xFFFF) + min(tie_rank, take_eq);
            for (int e = e0; e < e1; ++e) {
                const uint32_t key = sh.buf_key[e];
                if (key > thr || (key == thr && tie_rank++ < take_eq))
                    out[pos++] = sh.buf_id[e];
            }
            written = (sums & 0xFFFF) + min(sums >> 16, take_eq);
            done = true;
        }
    }

    if (!done) {
        // ---- exact fallback: streaming radix select over the row
        int above;
        thr = select_global(sh, sc, len, cur, forced, k, &above);
        take_eq = k - above;
    }
    if (!done || take_all) {
        // ---- ordered compaction over the row; thread t handles ids [tile + 8t, tile + 8t + 8)
        int eq_seen = 0;
        for (int tile = 0; tile < len; tile += kSelThreads * kSelBatch) {
            const int i0 = tile + tid * kSelBatch;
            unsigned gt_bits = 0, eq_bits = 0;
#pragma unroll
            for (int e = 0; e < kSelBatch; ++e) {
                const int i = i0 + e;
                const bool valid = i < len && !(forced && i == cur);
                const uint32_t key = valid ? score_key(sc[i]) : 0u;
                if (valid && (take_all || key > thr))
                    gt_bits |= 1u << e;
                if (valid && !take_all && key == thr)
                    eq_bits |= 1u << e;
            }
            int eq_total, take_total;
            const int eq_before = block_excl_sum(__popc(eq_bits), sh.cnt, &eq_total);
            unsigned take_bits = gt_bits;          // ties kept in id order up to take_eq
            int eq_idx = eq_seen + eq_before;
#pragma unroll
            for (int e = 0; e < kSelBatch; ++e)
                if ((eq_bits >> e) & 1u) {
                    if (eq_idx < take_eq)
                        take_bits |= 1u << e;
                    ++eq_idx;
                }
            int pos = base + written + block_excl_sum(__popc(take_bits), sh.cnt, &take_total);
#pragma unroll
            for (int e = 0; e < kSelBatch; ++e)
                if ((take_bits >> e) & 1u)
                    out[pos++] = i0 + e;
            written += take_total;
            eq_seen += eq_total;
        }
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

cudaError_t ensure_select_smem()
{
    static std::mutex mu;
    static bool raised[256] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 256 && raised[dev])
        return cudaSuccess;
    e = cudaFuncSetAttribute(sda_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(SelShared)));
    if (e == cudaSuccess)   // all of the unified L1/shared storage as shared: 4 CTAs per SM fit
        e = cudaFuncSetAttribute(sda_select_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess && dev >= 0 && dev < 256)
        raised[dev] = true;
    return e;
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
    if (rows > INT32_MAX || n_cols > INT32_MAX - kFilterStep)
        return SDA_ERR_UNSUPPORTED;
    if (rows == 0)
        return SDA_OK;
    if (!scores->data || !current->data || !regions->data)
        return SDA_ERR_INVALID;
    if (ensure_select_smem() != cudaSuccess)
        return SDA_ERR_CUDA;
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
    cfg.dynamicSmemBytes = sizeof(SelShared);
    cfg.stream = static_cast<cudaStream_t>(stream);
    return cudaLaunchKernelEx(&cfg, sda_select_kernel, prm) == cudaSuccess ? SDA_OK : SDA_ERR_CUDA;
}
