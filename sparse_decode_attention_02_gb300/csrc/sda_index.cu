// Indexer decode scores for sparse decode on GB300 (sm_103a).
//
// The adapter page "vllm.models.step5.nvidia.flashinfer_sparse" scores the
// 8-token regions of every decode row with `decode_logits` (fast path
// `decode_summary_scores`) before `select_regions` picks the row's top-k for
// `sparse_decode_attention`.  The page gives the operands — an FP8 E4M3 index
// query [tokens, G, 8, 256], fp32 head weights [tokens, G, 8], FP8 mean
// summaries [slots, G, 256] with one slot per 8-token region of every page —
// and names an FP8 paged MQA-logits kernel for the product, but prints no
// formula.  This kernel computes the reading declared in include/sdattn.h:
//     score[row, j] = sum_h w[h] * max(0, <q_h, m_j>)   for j <= pos / 8,
//     -inf for the remaining columns,
// with row = (token, g), pos the token's position and m_j the summary of
// region j of group g, found through the request's block-table row.
//
// Design.  A CTA takes one request and a chunk of its regions for a block of
// up to 4 KV groups, one warp per group (the groups' summaries of a slot are
// adjacent, so the CTA reads them as one run); with fewer groups per block the
// spare warps split the chunk.  Each warp streams 1024 regions of its group as
// 16-region tiles.  A tile (16 x 256 FP8 bytes, 4 KB) is copied with 16-byte
// cp.async into a 3- or 4-stage ring of the warp's own shared memory (see
// ring_tiles), XOR-swizzled per row so that ldmatrix reads are conflict-free.
// The product is an MMA with the regions as M (16) and the 8
// heads of one token as N: ldmatrix gives each lane 4 contiguous summary
// bytes per row, which serve both k16 steps of mma.sync m16n8k16 once the
// same byte-to-k permutation is applied to the query words (every k is still
// paired with itself); E4M3 bytes become fp16 exactly with
// cvt.rn.f16x2.e4m3x2, products accumulate in fp32.  The epilogue clamps at
// zero, weights, and sums the 8 heads across the lane quad.  The query_len
// tokens of a request share every summary tile, so each tile is read from HBM
// once per (request, group).  Bound: HBM — 256 summary bytes per region per
// (request, group) against 4096 flop per token.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "sdattn.h"

namespace {

constexpr int kIdxHeads = 8;
constexpr int kIdxDim = 256;          // bytes per head (E4M3) and per summary
constexpr int kRegionTokens = 8;
constexpr int kIdxWarps = 4;
constexpr int kIdxThreads = kIdxWarps * 32;
constexpr int kTile = 16;             // regions per tile (the MMA's M)
constexpr int kTilesPerWarp = 64;
constexpr int kWarpRegions = kTilesPerWarp * kTile;   // regions one warp streams
constexpr int kTileBytes = kTile * kIdxDim;
constexpr int kMaxQueryLen = 4;

// Tiles in a warp's ring and CTAs per SM, by tokens per request, as measured
// on 512 requests of 128K-256K tokens: a 3-tile ring (48 KB per CTA) at 4 CTAs
// per SM, except for 3 tokens, which ran 18 % slower that way than with a
// 4-tile ring (64 KB per CTA) at 3 CTAs per SM.
__host__ __device__ constexpr int ring_tiles(int ql) { return ql == 3 ? 4 : 3; }
__host__ __device__ constexpr int ctas_per_sm(int ql) { return ql == 3 ? 3 : 4; }
__host__ __device__ constexpr int index_smem_bytes(int ql) { return kIdxWarps * ring_tiles(ql) * kTileBytes; }
static_assert(ring_tiles(3) * kTile <= 64 && ring_tiles(1) * kTile <= 64,
              "the ring's row masks are packed into one 64-bit word");

struct IndexParams {
    const uint8_t *query;     // [tokens, G, 8, 256]
    int64_t q_s0, q_s1;
    const float *weights;     // [tokens, G, 8]
    int64_t w_s0, w_s1;
    const uint8_t *summaries; // [slots, G, 256]
    int64_t m_s0, n_slots;
    const int32_t *table;     // [reqs, width]
    int64_t bt_s0;
    int width;
    const int32_t *seq_lens;
    int64_t sl_s0;
    float *scores;            // [tokens * G, n_cols]
    int64_t sc_s0;
    int32_t *current;         // [tokens * G] or NULL
    int64_t cur_s0;
    int32_t *lengths;         // [tokens * G] or NULL
    int64_t len_s0;
    uint32_t *flags;          // workspace header or NULL
    int groups, block, n_cols;
    int chunks;               // CTAs per (request, group block)
};

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes)
{
    uint32_t r;
    const uint16_t v = static_cast<uint16_t>(two_bytes);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
    return r;
}

__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Shared-memory offset of 16-byte segment `seg` (0..15) of tile row `row`:
// rows are 256 bytes, segments XOR-swizzled by the row's low 3 bits so the 8
// rows of one ldmatrix matrix fall in 8 different 16-byte bank groups.
__device__ __forceinline__ uint32_t tile_offset(int row, int seg)
{
    return static_cast<uint32_t>(row * kIdxDim + ((seg ^ (row & 7)) << 4));
}

// QL = tokens per request, GB = groups per CTA (4, 2 or 1, dividing G; the
// 4 / GB warps of a group split the CTA's regions).  Each lane keeps, per
// token and 32-dim chunk kc, the query words w0 = bytes [32kc + 4t, +4) and
// w1 = bytes [32kc + 16 + 4t, +4) of head `gid` (lane = 4 gid + t).  For
// QL <= 2 they are held already converted to fp16 pairs.
template <int QL, int GB>
__global__ void __launch_bounds__(kIdxThreads, ctas_per_sm(QL)) sda_index_kernel(const IndexParams p)
{
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int kStages = ring_tiles(QL);
    constexpr bool kPreconv = QL <= 2;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, t4 = lane & 3;

    const int64_t unit = blockIdx.x;
    const int chunk = static_cast<int>(unit % p.chunks);
    const int64_t rest = unit / p.chunks;
    constexpr int kChunkRegions = (kIdxWarps / GB) * kWarpRegions;
    const int gblocks = p.groups / GB;
    const int g = static_cast<int>(rest % gblocks) * GB + warp % GB;
    const int sub = warp / GB;   // this warp's part of the chunk
    const int64_t req = rest / gblocks;

    const int64_t seq_len = p.seq_lens[req * p.sl_s0];
    int n_tok[QL];
    int n_max = 0;
#pragma unroll
    for (int i = 0; i < QL; ++i) {
        const int64_t pos = seq_len - QL + i;
        int64_t n = pos >= 0 ? pos / kRegionTokens + 1 : 0;
        if (n > p.n_cols)
            n = p.n_cols;
        n_tok[i] = static_cast<int>(n);
        n_max = n_tok[i] > n_max ? n_tok[i] : n_max;
        if (chunk == 0 && sub == 0 && lane == 0) {
            const int64_t row = (req * QL + i) * p.groups + g;
            if (p.current)
                p.current[row * p.cur_s0] = pos >= 0 ? static_cast<int32_t>(pos / kRegionTokens) : -1;
            if (p.lengths)
                p.lengths[row * p.len_s0] = static_cast<int32_t>(n);
        }
    }

    const int region0 = chunk * kChunkRegions + sub * kWarpRegions;
    int tiles = 0;   // tiles of this warp that hold scored regions
    if (region0 < n_max)
        tiles = min(kTilesPerWarp, (n_max - region0 + kTile - 1) / kTile);

    // Query words and head weights of the request's tokens.
    uint32_t qraw[kPreconv ? 1 : QL][8][2];
    uint32_t qcv[kPreconv ? QL : 1][8][4];
    float wlo[QL], whi[QL];
#pragma unroll
    for (int i = 0; i < QL; ++i) {
        const int64_t tok = req * QL + i;
        const float *w = p.weights + tok * p.w_s0 + g * p.w_s1 + 2 * t4;
        wlo[i] = w[0];
        whi[i] = w[1];
        if (tiles == 0)
            continue;
        const uint8_t *q = p.query + tok * p.q_s0 + g * p.q_s1 + gid * kIdxDim + 4 * t4;
#pragma unroll
        for (int kc = 0; kc < 8; ++kc) {
            const uint32_t w0 = __ldg(reinterpret_cast<const uint32_t *>(q + 32 * kc));
            const uint32_t w1 = __ldg(reinterpret_cast<const uint32_t *>(q + 32 * kc + 16));
            if constexpr (kPreconv) {
                qcv[i][kc][0] = e4m3x2_to_f16x2(w0);
                qcv[i][kc][1] = e4m3x2_to_f16x2(w0 >> 16);
                qcv[i][kc][2] = e4m3x2_to_f16x2(w1);
                qcv[i][kc][3] = e4m3x2_to_f16x2(w1 >> 16);
            } else {
                qraw[i][kc][0] = w0;
                qraw[i][kc][1] = w1;
            }
        }
    }

    uint8_t *ring = smem + warp * (kStages * kTileBytes);
    const uint32_t ring_s = smem_u32(ring);
    const int per_page = p.block / kRegionTokens;
    const uint8_t *msum = p.summaries + static_cast<int64_t>(g) * kIdxDim;
    const int32_t *trow = p.table + req * p.bt_s0;

    // Issue the copies of tile `tt` into its ring slot; returns the 16-bit
    // mask of rows whose summary exists (the lane-uniform result).
    auto issue = [&](int tt) -> uint32_t {
        const int base = region0 + tt * kTile;
        int64_t slot = -1;
        if (lane < kTile) {
            const int j = base + lane;
            if (j < n_max) {
                const int64_t tok0 = static_cast<int64_t>(j) * kRegionTokens;
                const int64_t col = tok0 / p.block;
                bool ok = col < p.width;
                if (ok) {
                    const int64_t page = trow[col];
                    slot = page * per_page + (tok0 % p.block) / kRegionTokens;
                    ok = page >= 0 && slot < p.n_slots;
                }
                if (!ok) {
                    slot = -1;
                    if (p.flags)
                        atomicOr(p.flags, SDA_FLAG_BOUNDS);
                }
            }
        }
        const uint32_t valid = __ballot_sync(0xffffffffu, slot >= 0) & 0xffffu;
        const uint32_t dst0 = ring_s + (tt % kStages) * kTileBytes;
        const int seg = lane & 15;
#pragma unroll
        for (int i = 0; i < kTile / 2; ++i) {
            const int row = 2 * i + (lane >> 4);
            const int64_t s = __shfl_sync(0xffffffffu, slot, row);
            if (s >= 0)
                cp_async16(dst0 + tile_offset(row, seg), msum + s * p.m_s0 + seg * 16);
        }
        return valid;
    };

    uint64_t vm = 0;   // the 16-bit row masks of the tiles in flight, by ring slot
#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
        if (s < tiles)
            vm |= static_cast<uint64_t>(issue(s)) << (16 * s);
        cp_async_commit();
    }

    // ldmatrix x4: matrix mi = lane / 8 is (rows 0-7 | rows 8-15) x
    // (segment 2kc | 2kc + 1); lane gets bytes [4 t4, +4) of row gid of each.
    const int lrow = ((lane >> 3) & 1) * 8 + (lane & 7);
    const int lseg = lane >> 4;
    float *srow[QL];
#pragma unroll
    for (int i = 0; i < QL; ++i)
        srow[i] = p.scores + ((req * QL + i) * p.groups + g) * p.sc_s0;

    for (int tt = 0; tt < kTilesPerWarp; ++tt) {
        const int nx = tt + kStages - 1;
        if (nx < tiles) {
            const int sl = nx % kStages;
            vm = (vm & ~(0xffffull << (16 * sl))) | (static_cast<uint64_t>(issue(nx)) << (16 * sl));
        }
        cp_async_commit();
        const int base = region0 + tt * kTile;
        if (base >= p.n_cols)
            break;
        if (tt >= tiles) {   // nothing scored in this tile: -inf for every token
            if (lane < kTile && base + lane < p.n_cols) {
#pragma unroll
                for (int i = 0; i < QL; ++i)
                    srow[i][base + lane] = -INFINITY;
            }
            continue;
        }
        cp_async_wait<kStages - 1>();
        __syncwarp();
        const uint32_t valid = static_cast<uint32_t>(vm >> (16 * (tt % kStages))) & 0xffffu;
        const uint32_t tbase = ring_s + (tt % kStages) * kTileBytes;
        float acc[QL][4];
#pragma unroll
        for (int i = 0; i < QL; ++i)
            acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
        for (int kc = 0; kc < 8; ++kc) {
            uint32_t m0, m1, m2, m3;
            ldsm_x4(tbase + tile_offset(lrow, 2 * kc + lseg), m0, m1, m2, m3);
            // k step over segment 2kc: bytes (4t, 4t+1) are k (2t, 2t+1) and
            // bytes (4t+2, 4t+3) are k (2t+8, 2t+9), for A and B alike.
            uint32_t a0 = e4m3x2_to_f16x2(m0), a1 = e4m3x2_to_f16x2(m1);
            uint32_t a2 = e4m3x2_to_f16x2(m0 >> 16), a3 = e4m3x2_to_f16x2(m1 >> 16);
#pragma unroll
            for (int i = 0; i < QL; ++i) {
                if constexpr (kPreconv)
                    mma_f16(acc[i], a0, a1, a2, a3, qcv[i][kc][0], qcv[i][kc][1]);
                else
                    mma_f16(acc[i], a0, a1, a2, a3, e4m3x2_to_f16x2(qraw[i][kc][0]),
                            e4m3x2_to_f16x2(qraw[i][kc][0] >> 16));
            }
            a0 = e4m3x2_to_f16x2(m2);
            a1 = e4m3x2_to_f16x2(m3);
            a2 = e4m3x2_to_f16x2(m2 >> 16);
            a3 = e4m3x2_to_f16x2(m3 >> 16);
#pragma unroll
            for (int i = 0; i < QL; ++i) {
                if constexpr (kPreconv)
                    mma_f16(acc[i], a0, a1, a2, a3, qcv[i][kc][2], qcv[i][kc][3]);
                else
                    mma_f16(acc[i], a0, a1, a2, a3, e4m3x2_to_f16x2(qraw[i][kc][1]),
                            e4m3x2_to_f16x2(qraw[i][kc][1] >> 16));
            }
        }
        __syncwarp();   // the slot is refilled by the next iteration's copies
        // acc: [0], [1] = row gid, heads 2t, 2t+1; [2], [3] = row gid + 8.
        const int r = gid + 8 * t4;
        const int j = base + r;
#pragma unroll
        for (int i = 0; i < QL; ++i) {
            float lo = wlo[i] * fmaxf(acc[i][0], 0.f) + whi[i] * fmaxf(acc[i][1], 0.f);
            float hi = wlo[i] * fmaxf(acc[i][2], 0.f) + whi[i] * fmaxf(acc[i][3], 0.f);
            lo += __shfl_xor_sync(0xffffffffu, lo, 1);
            hi += __shfl_xor_sync(0xffffffffu, hi, 1);
            lo += __shfl_xor_sync(0xffffffffu, lo, 2);
            hi += __shfl_xor_sync(0xffffffffu, hi, 2);
            if (t4 < 2 && j < p.n_cols) {
                const bool scored = j < n_tok[i] && ((valid >> r) & 1u);
                srow[i][j] = scored ? (t4 ? hi : lo) : -INFINITY;
            }
        }
    }
}

cudaError_t ensure_index_smem(const void *kernel, int slot, int smem_bytes)
{
    static std::mutex mu;
    static bool raised[kMaxQueryLen * 3][256] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 256 && raised[slot][dev])
        return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e == cudaSuccess)   // all of the unified L1/shared storage as shared: ctas_per_sm CTAs fit
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess && dev >= 0 && dev < 256)
        raised[slot][dev] = true;
    return e;
}

bool dims_ok(const sda_tensor *t, int ndim)
{
    if (!t || t->ndim != ndim)
        return false;
    for (int i = 0; i < ndim; ++i)
        if (t->shape[i] < 0)
            return false;
    return true;
}

bool is_bytes(const sda_tensor *t)
{
    return t->dtype == SDA_DTYPE_FP8_E4M3 || t->dtype == SDA_DTYPE_UINT8;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" sda_status sparse_decode_summary_scores(
    const sda_tensor *query, const sda_tensor *weights, const sda_tensor *summaries,
    const sda_tensor *block_table, const sda_tensor *seq_lens, int block_size, int query_len,
    const sda_tensor *scores, const sda_tensor *current, const sda_tensor *lengths, void *workspace,
    size_t workspace_bytes, void *stream)
{
    if (!dims_ok(query, 4) || !dims_ok(weights, 3) || !dims_ok(summaries, 3) ||
        !dims_ok(block_table, 2) || !dims_ok(seq_lens, 1) || !dims_ok(scores, 2))
        return SDA_ERR_INVALID;
    if (query_len < 1 || block_size < kRegionTokens || block_size % kRegionTokens)
        return SDA_ERR_INVALID;
    const int64_t tokens = query->shape[0], groups = query->shape[1];
    if (!is_bytes(query) || query->shape[2] != kIdxHeads || query->shape[3] != kIdxDim ||
        query->stride[3] != 1 || query->stride[2] != kIdxDim || groups < 1)
        return SDA_ERR_INVALID;
    if (weights->dtype != SDA_DTYPE_FP32 || weights->shape[0] != tokens ||
        weights->shape[1] != groups || weights->shape[2] != kIdxHeads || weights->stride[2] != 1)
        return SDA_ERR_INVALID;
    if (!is_bytes(summaries) || summaries->shape[1] != groups || summaries->shape[2] != kIdxDim ||
        summaries->stride[2] != 1 || summaries->stride[1] != kIdxDim)
        return SDA_ERR_INVALID;
    if (block_table->dtype != SDA_DTYPE_INT32 ||
        (block_table->shape[1] > 1 && block_table->stride[1] != 1))
        return SDA_ERR_INVALID;
    if (tokens % query_len)
        return SDA_ERR_INVALID;
    const int64_t reqs = tokens / query_len;
    if (seq_lens->dtype != SDA_DTYPE_INT32 || seq_lens->shape[0] < reqs ||
        block_table->shape[0] < reqs)
        return SDA_ERR_INVALID;
    const int64_t rows = tokens * groups, n_cols = scores->shape[1];
    if (scores->dtype != SDA_DTYPE_FP32 || scores->shape[0] != rows ||
        (n_cols > 1 && scores->stride[1] != 1))
        return SDA_ERR_INVALID;
    const bool has_cur = current && current->data, has_len = lengths && lengths->data;
    if (has_cur && (!dims_ok(current, 1) || current->dtype != SDA_DTYPE_INT32 ||
                    current->shape[0] != rows))
        return SDA_ERR_INVALID;
    if (has_len && (!dims_ok(lengths, 1) || lengths->dtype != SDA_DTYPE_INT32 ||
                    lengths->shape[0] != rows))
        return SDA_ERR_INVALID;
    if (workspace && ((reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < 256))
        return SDA_ERR_WORKSPACE;
    if (query_len > kMaxQueryLen)
        return SDA_ERR_UNSUPPORTED;
    // 16-byte copies and 4-byte query loads.
    if (query->stride[0] % 16 || query->stride[1] % 16 || summaries->stride[0] % 16)
        return SDA_ERR_UNSUPPORTED;
    // The warps of a CTA take the same regions of up to 4 groups (their
    // summaries are adjacent in memory), or split the regions of fewer.
    const int gblock = groups % 4 == 0 ? 4 : (groups % 2 == 0 ? 2 : 1);
    const int chunk_regions = (kIdxWarps / gblock) * kWarpRegions;
    const int64_t chunks = n_cols > 0 ? (n_cols + chunk_regions - 1) / chunk_regions : 1;
    if (n_cols > INT32_MAX - chunk_regions || block_table->shape[1] > INT32_MAX ||
        block_size > INT32_MAX / 2 || groups > INT32_MAX || chunks * (groups / gblock) * reqs > INT32_MAX)
        return SDA_ERR_UNSUPPORTED;
    if (rows == 0)
        return SDA_OK;
    if (!query->data || !weights->data || !summaries->data || !block_table->data || !seq_lens->data ||
        (n_cols > 0 && !scores->data))
        return SDA_ERR_INVALID;
    if (!aligned16(query->data) || !aligned16(summaries->data))
        return SDA_ERR_UNSUPPORTED;

    IndexParams prm;
    prm.query = static_cast<const uint8_t *>(query->data);
    prm.q_s0 = query->stride[0];
    prm.q_s1 = query->stride[1];
    prm.weights = static_cast<const float *>(weights->data);
    prm.w_s0 = weights->stride[0];
    prm.w_s1 = weights->stride[1];
    prm.summaries = static_cast<const uint8_t *>(summaries->data);
    prm.m_s0 = summaries->stride[0];
    prm.n_slots = summaries->shape[0];
    prm.table = static_cast<const int32_t *>(block_table->data);
    prm.bt_s0 = block_table->stride[0];
    prm.width = static_cast<int>(block_table->shape[1]);
    prm.seq_lens = static_cast<const int32_t *>(seq_lens->data);
    prm.sl_s0 = seq_lens->stride[0];
    prm.scores = static_cast<float *>(const_cast<void *>(scores->data));
    prm.sc_s0 = scores->stride[0];
    prm.current = has_cur ? static_cast<int32_t *>(const_cast<void *>(current->data)) : nullptr;
    prm.cur_s0 = has_cur ? current->stride[0] : 0;
    prm.lengths = has_len ? static_cast<int32_t *>(const_cast<void *>(lengths->data)) : nullptr;
    prm.len_s0 = has_len ? lengths->stride[0] : 0;
    prm.flags = static_cast<uint32_t *>(workspace);
    prm.groups = static_cast<int>(groups);
    prm.block = block_size;
    prm.n_cols = static_cast<int>(n_cols);
    prm.chunks = static_cast<int>(chunks);

#define SDA_INDEX_KERNELS(QL)                                                   \
    {reinterpret_cast<const void *>(sda_index_kernel<QL, 1>),                   \
     reinterpret_cast<const void *>(sda_index_kernel<QL, 2>),                   \
     reinterpret_cast<const void *>(sda_index_kernel<QL, 4>)}
    const void *kernels[kMaxQueryLen][3] = {SDA_INDEX_KERNELS(1), SDA_INDEX_KERNELS(2),
                                            SDA_INDEX_KERNELS(3), SDA_INDEX_KERNELS(4)};
#undef SDA_INDEX_KERNELS
    const int gb_slot = gblock == 4 ? 2 : gblock - 1;
    const void *kernel = kernels[query_len - 1][gb_slot];
    if (ensure_index_smem(kernel, (query_len - 1) * 3 + gb_slot, index_smem_bytes(query_len)) != cudaSuccess)
        return SDA_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(chunks * (groups / gblock) * reqs));
    cfg.blockDim = dim3(kIdxThreads);
    cfg.dynamicSmemBytes = index_smem_bytes(query_len);
    cfg.stream = static_cast<cudaStream_t>(stream);
    void *args[] = {&prm};
    return cudaLaunchKernelExC(&cfg, kernel, args) == cudaSuccess ? SDA_OK : SDA_ERR_CUDA;
}
