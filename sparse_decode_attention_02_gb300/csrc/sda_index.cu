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
// Design.  Two kernels compute it.  Pages of a multiple of 64 tokens (every
// workload here) take the tensor-core kernel, sda_index_tc_kernel: persistent
// CTAs, one per SM, each with an equal share of all 128-row tiles; TMA boxes
// of whole pages (8 summary slots x 256 bytes x a block of up to 4 groups)
// into a shared-memory ring; tcgen05.mma kind::f8f6f4 on the raw E4M3 bytes,
// regions x (tokens, groups, heads), fp32 accumulators in tensor memory; an
// epilogue of eight warps reading them back with tcgen05.ld (details above
// the kernel).  Smaller pages take sda_index_kernel, the mma.sync design below.
//
// sda_index_kernel.  A CTA takes one request and a chunk of its regions for a
// block of up to 4 KV groups, one warp per group (the groups' summaries of a
// slot are adjacent, so the CTA reads them as one run); with fewer groups per
// block the spare warps split the chunk.  Each warp streams 1024 regions of
// its group as 16-region tiles.  A tile (16 x 256 FP8 bytes, 4 KB) is copied
// with 16-byte cp.async into a 3- or 4-stage ring of the warp's own shared
// memory (see ring_tiles), XOR-swizzled per row so that ldmatrix reads are
// conflict-free.  The product is an MMA with the regions as M (16) and the 8
// heads of one token as N: ldmatrix gives each lane 4 contiguous summary
// bytes per row, which serve both k16 steps of mma.sync m16n8k16 once the
// same byte-to-k permutation is applied to the query words (every k is still
// paired with itself); E4M3 bytes become fp16 exactly with
// cvt.rn.f16x2.e4m3x2, products accumulate in fp32.  The epilogue clamps at
// zero, weights, and sums the 8 heads across the lane quad.
//
// Both read each summary from HBM once per (request, group): the query_len
// tokens of a request share it.  Bound: HBM — 256 summary bytes per region
// per (request, group) against 4096 flop per token.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "sdattn.h"

// The process-wide limit of the kernels' pipeline waits (set with
// sparse_decode_set_wait_limit_ns).
uint64_t sda_wait_limit_ns();

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

// ---------------------------------------------------------------------------
// Tensor-core (tcgen05) variant, for pages of a multiple of 64 tokens.
//
// Work: every (request, block of GB = 4, 2 or 1 groups) row set is cut into
// tiles of 128 MMA rows = 128 / (8 GB) runs of 8 consecutive regions, each run
// with all GB groups.  One persistent CTA per SM takes an equal contiguous
// range of all these tiles (found with one scan of seq_lens), and walks it in
// pieces of at most 16 tiles of one row set.  Warp 0 resolves a piece's pages
// through the block table (the next piece's entries load while this one is
// copied) and copies each run with one 5-D TMA box (8 summary slots x both
// 128-byte K halves x GB groups of one page, 128-byte swizzle, 2 GB KB) into a
// ring that runs on across pieces; the box lands as [group][K half][slot][128
// bytes], so K half h of the tile is a K-major operand whose 8-row core groups
// (run, group) sit 2 KB apart.  One thread of warp 1 keeps two query buffers,
// loading the next piece's query heads with TMA (rows (token, group, head),
// N = 8 GB query_len rounded up to 16, 256 bytes each) while the current one
// runs, and issues tcgen05.mma kind::f8f6f4 on the raw E4M3 bytes: A = the
// tile (M = 128), B = the query rows of all GB groups, K = 256 in 8 steps of
// 32, fp32 accumulators in tensor memory (up to 8 buffers, allocated once per
// CTA).  Row m of an accumulator holds its region's products with every
// group's heads; eight epilogue warps, two per 32-lane quarter of tensor
// memory (one for the first half of the tokens, one for the rest), read them
// with tcgen05.ld (one region and group per thread), keep the columns of
// their own group, clamp at zero, weight, sum the 8 heads per token and store
// the scores.  No conversions and no per-token MMAs: query_len 1-4 stream the
// summaries at nearly the same cost (the MMAs the other groups' columns cost
// are cheap next to the stream).
// ---------------------------------------------------------------------------

constexpr int kTcM = 128;                    // MMA rows per tile
constexpr int kTcTileBytes = kTcM * kIdxDim; // 32 KB
constexpr int kTcPieceTiles = 16;            // tiles per piece
constexpr int kTcEpiWarps = 8;               // two per tensor-memory lane quarter
constexpr int kTcThreads = 64 + 32 * kTcEpiWarps;   // producer, MMA, epilogue warps
constexpr int kTcCtasPerSm = 1;
constexpr uint64_t kTcDrainNs = 1000000000ull;

// Per (query_len, groups per block): MMA N, accumulators, tensor-memory
// columns (a power of two), ring stages and shared-memory layout.
template <int QL, int GB>
struct TcCfg {
    static constexpr int kN = (8 * GB * QL + 15) / 16 * 16;
    static constexpr int kAcc = 512 / kN < 8 ? 512 / kN : 8;
    static constexpr int kTmemCols = kAcc * kN <= 32 ? 32 : kAcc * kN <= 64 ? 64 : kAcc * kN <= 128 ? 128
                                   : kAcc * kN <= 256 ? 256 : 512;
    static constexpr int kRuns = kTcM / (8 * GB);           // 8-region runs per tile
    static constexpr int kRegions = 8 * kRuns;              // regions per tile
    static constexpr int kPieceRuns = kTcPieceTiles * kRuns;
    static constexpr int kQBuf = kN * kIdxDim;              // one query buffer: [2 halves][N rows][128 B]
    static constexpr int kMisc = 8 * kPieceRuns + 8 * 64 + 64;
    static constexpr int kStages0 = (227 * 1024 - 1024 - 2 * kQBuf - kMisc) / kTcTileBytes;
    static constexpr int kStages = kStages0 > 6 ? 6 : kStages0;
    // offsets from the 1 KB aligned base
    static constexpr int kQ = kStages * kTcTileBytes;
    static constexpr int kTbuf = kQ + 2 * kQBuf;            // two buffers of a piece's page ids
    static constexpr int kBar = kTbuf + 8 * kPieceRuns;
    // full[S] empty[S] tfull[A] tempty[A] qfull[2] qempty[2] tbfull[2] tbfree[2] mdone
    static constexpr int kStart = kBar + 8 * (2 * kStages + 2 * kAcc + 9);   // the CTA's range: 4 x int64
    static constexpr int kTmemSlot = kStart + 32;
    static constexpr int kAbort = kTmemSlot + 4;
    static constexpr int kAlloc = kAbort + 4 + 1024;
    static_assert(kStages >= 3, "ring depth");
    static_assert(kAcc * kN <= 512 && kQBuf % 1024 == 0 && kAlloc <= 227 * 1024, "tc resources");
};

struct IndexTcParams {
    const float *weights;     // [tokens, G, 8]
    int64_t w_s0, w_s1;
    const int32_t *table;     // [reqs, width]
    int64_t bt_s0;
    int width;
    const int32_t *seq_lens;
    int64_t sl_s0;
    float *scores;            // [tokens * G, n_cols]
    int64_t sc_s0;
    int32_t *current;
    int64_t cur_s0;
    int32_t *lengths;
    int64_t len_s0;
    uint32_t *flags;          // workspace header or NULL
    int64_t pages;            // pages the summaries hold (slots / per_page)
    int64_t reqs;
    unsigned long long wait_ns;
    int groups, gblocks, block, n_cols;
    int per_page;             // summary slots (regions) per page
};

// The scored-region count and current region of each of request r's tokens,
// and its tiles: at least one, so that every row set has a tile whose piece
// writes its -inf tail, `current` and `lengths`.
template <int QL, int GB>
struct TcReq {
    int n_tok[QL];   // scored regions of each token
    int cur[QL];     // the region holding each token (-1 before the sequence starts)
    int n_max, tiles;
    TcReq() = default;
    __device__ TcReq(const IndexTcParams &p, int64_t r)
    {
        const int64_t seq_len = p.seq_lens[r * p.sl_s0];
        n_max = 0;
#pragma unroll
        for (int i = 0; i < QL; ++i) {
            const int64_t pos = seq_len - QL + i;
            const int64_t n = pos >= 0 ? pos / kRegionTokens + 1 : 0;
            n_tok[i] = static_cast<int>(n < p.n_cols ? n : p.n_cols);
            cur[i] = pos >= 0 ? static_cast<int>(pos / kRegionTokens) : -1;
            n_max = max(n_max, n_tok[i]);
        }
        tiles = max(1, (n_max + TcCfg<QL, GB>::kRegions - 1) / TcCfg<QL, GB>::kRegions);
    }
};

// A piece: tiles [t0, t0 + nt) of one (request, group block) row set.
template <int QL, int GB>
struct TcPiece {
    int64_t req;
    int gb0, t0, nt;
    bool first, last;        // holds the row set's first / last tile
    TcReq<QL, GB> rq;
    __device__ int lo() const { return t0 * TcCfg<QL, GB>::kRegions; }
};

// Walks a CTA's tile range piece by piece (every role keeps its own cursor).
template <int QL, int GB>
struct TcCursor {
    int64_t r, remaining;
    int gbk, t;
    TcReq<QL, GB> rq;
    __device__ TcCursor(const IndexTcParams &p, const int64_t *start)
        : r(start[0]), remaining(start[3]), gbk(static_cast<int>(start[1])), t(static_cast<int>(start[2])),
          rq(p, start[0] < p.reqs ? start[0] : 0) {}
    __device__ bool next(const IndexTcParams &p, TcPiece<QL, GB> &pc)
    {
        if (remaining <= 0)
            return false;
        const int nt = static_cast<int>(min(static_cast<int64_t>(min(kTcPieceTiles, rq.tiles - t)), remaining));
        pc.req = r;
        pc.gb0 = gbk * GB;
        pc.t0 = t;
        pc.nt = nt;
        pc.first = t == 0;
        pc.last = t + nt == rq.tiles;
        pc.rq = rq;
        remaining -= nt;
        t += nt;
        if (t == rq.tiles) {
            t = 0;
            if (++gbk == p.gblocks) {
                gbk = 0;
                ++r;
                if (remaining > 0)
                    rq = TcReq<QL, GB>(p, r);
            }
        }
        return true;
    }
};

__device__ __forceinline__ void tc_mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void tc_mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void tc_mbar_arrive(uint32_t bar)
{
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool tc_mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t tc_now_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for the phase of `bar` with the given parity; false after limit_ns,
// or at once when another role of the CTA has given up (*abort, if given).
__device__ __forceinline__ bool tc_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                        const volatile int *abort = nullptr)
{
    if (tc_mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = tc_now_ns();
    for (;;) {
        if (tc_mbar_try_wait(bar, parity))
            return true;
        if ((abort && *abort) || tc_now_ns() - t0 > limit_ns)
            return false;
    }
}

__device__ __forceinline__ void tc_tma_5d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2, int c3,
                                          int c4, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar)
        : "memory");
}

// Shared-memory matrix descriptor of a K-major operand with 128-byte swizzle:
// rows of 128 bytes in 8-row core groups of 1024 bytes, `sbo` bytes apart
// (start address in 16-byte units in bits 0-13, leading offset 16 bytes
// (unused for this layout) in 16-29, stride `sbo` in 16-byte units in 32-45,
// descriptor version 1 in 46-47, swizzle mode 2 = 128-byte in 61-63).
__device__ __forceinline__ uint64_t tc_desc_sw128(uint32_t saddr, uint32_t sbo)
{
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(sbo >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}

// Instruction descriptor of tcgen05.mma kind::f8f6f4: D fp32 (bits 4-5 = 1),
// A and B E4M3 (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t tc_idesc(int n, int m)
{
    return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 lanes x 16 columns of fp32 from tensor memory (thread t: lane base + t),
// into r; the caller waits with tcgen05.wait::ld before reading them.
__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t *r)
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
        "%13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// The epilogue of one warp of sda_index_tc_kernel for tokens [I0, I1): per
// tile, the accumulator columns of those tokens (column n: token n / (8 GB),
// group n / 8 % GB, head n % 8) for this thread's row (region and group),
// clamped at zero, weighted and summed over the 8 heads of its own group.
template <int QL, int GB, int I0, int I1>
__device__ __forceinline__ void tc_epilogue(const IndexTcParams &p, uint32_t tmem, const int32_t *tbuf,
                                            const int64_t *start, uint32_t tfull_bar, uint32_t tempty_bar,
                                            uint32_t tbfull_bar, uint32_t tbfree_bar, volatile int *abort)
{
    using C = TcCfg<QL, GB>;
    constexpr int N = C::kN, A = C::kAcc, R = C::kRuns;
    constexpr int kC0 = I0 * 8 * GB / 16 * 16;                       // first column chunk loaded
    constexpr int kC1 = I1 > I0 ? (I1 * 8 * GB + 15) / 16 * 16 : kC0;  // end of the chunks
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3;
    const int m = 32 * q + lane;
    const int run = m / (8 * GB), gl = (m / 8) % GB, slot = m % 8;
    const int et = threadIdx.x - 64;   // 0 .. 32 kTcEpiWarps - 1 among the epilogue threads
    TcCursor<QL, GB> cur(p, start);
    TcPiece<QL, GB> pc;
    int done = 0;                      // tiles handled
    for (int a = 0; cur.next(p, pc); ++a) {
        const int g = pc.gb0 + gl;
        if (pc.first && et < GB) {
#pragma unroll
            for (int i = 0; i < QL; ++i) {
                const int64_t row = (pc.req * QL + i) * p.groups + pc.gb0 + et;
                if (p.current)
                    p.current[row * p.cur_s0] = pc.rq.cur[i];
                if (p.lengths)
                    p.lengths[row * p.len_s0] = pc.rq.n_tok[i];
            }
        }
        float *srow[QL];
        float wt[QL][8];
#pragma unroll
        for (int i = I0; i < I1; ++i) {
            srow[i] = p.scores + ((pc.req * QL + i) * p.groups + g) * p.sc_s0;
#pragma unroll
            for (int h = 0; h < 8; ++h)
                wt[i][h] = p.weights[(pc.req * QL + i) * p.w_s0 + g * p.w_s1 + h];
        }
        // this piece's page ids (written by the producer into tbuf[a & 1]);
        // every lane waits (acquires) before reading them
        const int b = a & 1;
        if (!__all_sync(~0u, tc_wait(tbfull_bar + 8 * b, (a >> 1) & 1, p.wait_ns, abort))) {
            if (lane == 0) {
                *abort = 1;
                if (p.flags)
                    atomicOr(p.flags, SDA_FLAG_TIMEOUT);
            }
            return;
        }
        const int32_t *tb = tbuf + b * C::kPieceRuns;
        for (int t = 0; t < pc.nt; ++t, ++done) {
            const int acc = done % A;
            if (!__all_sync(~0u, tc_wait(tfull_bar + 8 * acc, (done / A) & 1, p.wait_ns, abort))) {
                if (lane == 0) {
                    *abort = 1;
                    if (p.flags)
                        atomicOr(p.flags, SDA_FLAG_TIMEOUT);
                }
                return;
            }
            tc_fence_after();
            float sc[QL];
#pragma unroll
            for (int i = 0; i < QL; ++i)
                sc[i] = 0.0f;
            if constexpr (kC1 > kC0) {
                uint32_t d[kC1 - kC0];   // all column loads in flight, one wait
#pragma unroll
                for (int c0 = kC0; c0 < kC1; c0 += 16)
                    tc_ld16(tmem + (static_cast<uint32_t>(32 * q) << 16) + acc * N + c0, d + (c0 - kC0));
                tc_wait_ld();
#pragma unroll
                for (int n = kC0; n < kC1; ++n) {
                    const int i = n / (8 * GB), gn = (n / 8) % GB, h = n % 8;
                    if (i >= I0 && i < I1 && gn == gl)
                        sc[i] += wt[i][h] * fmaxf(__uint_as_float(d[n - kC0]), 0.0f);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                tc_mbar_arrive(tempty_bar + 8 * acc);
            const int j = pc.lo() + t * C::kRegions + 8 * run + slot;
            const bool valid = tb[t * R + run] >= 0;   // an unresolvable page's rows were not copied
#pragma unroll
            for (int i = I0; i < I1; ++i)
                if (j < p.n_cols)
                    srow[i][j] = (valid && j < pc.rq.n_tok[i]) ? sc[i] : -INFINITY;
        }
        __syncwarp();
        if (lane == 0)
            tc_mbar_arrive(tbfree_bar + 8 * b);    // this warp is done with the piece's ids
        if (pc.last) {
            // the row set's columns past its last tile: -inf for every token and group
            const int from = (pc.t0 + pc.nt) * C::kRegions;
            const int width = p.n_cols - from;
            for (int e2 = et; e2 < GB * (width > 0 ? width : 0); e2 += 32 * kTcEpiWarps) {
                const int gg = pc.gb0 + e2 / width, j = from + e2 % width;
#pragma unroll
                for (int i = 0; i < QL; ++i)
                    p.scores[((pc.req * QL + i) * p.groups + gg) * p.sc_s0 + j] = -INFINITY;
            }
        }
    }
}

template <int QL, int GB>
__global__ void __launch_bounds__(kTcThreads, kTcCtasPerSm)
    sda_index_tc_kernel(const __grid_constant__ CUtensorMap smap, const __grid_constant__ CUtensorMap qmap,
                        const __grid_constant__ IndexTcParams p)
{
    using C = TcCfg<QL, GB>;
    constexpr int N = C::kN, S = C::kStages, A = C::kAcc, R = C::kRuns;
    constexpr uint32_t kIdesc = tc_idesc(N, kTcM);
    constexpr uint32_t kQBoxBytes = 8 * GB * QL * 128;   // one K half of a piece's query rows
    constexpr uint32_t kBoxBytes = GB * 2 * 8 * 128;      // one run: GB groups x 2 halves x 8 slots
    extern __shared__ uint8_t tc_smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(sm);
    const uint32_t full_bar = sbase + C::kBar;
    const uint32_t empty_bar = full_bar + 8 * S;
    const uint32_t tfull_bar = empty_bar + 8 * S;
    const uint32_t tempty_bar = tfull_bar + 8 * A;
    const uint32_t qfull_bar = tempty_bar + 8 * A;
    const uint32_t qempty_bar = qfull_bar + 16;
    const uint32_t tbfull_bar = qempty_bar + 16;
    const uint32_t tbfree_bar = tbfull_bar + 16;
    const uint32_t mdone_bar = tbfree_bar + 16;
    int32_t *tbuf = reinterpret_cast<int32_t *>(sm + C::kTbuf);     // [2][kPieceRuns]
    int64_t *start = reinterpret_cast<int64_t *>(sm + C::kStart);   // r, group block, tile, tiles
    volatile int *abort = reinterpret_cast<volatile int *>(sm + C::kAbort);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- set-up: barriers and this CTA's tile range (warp 0), tensor memory (warp 1)
    if (warp == 0) {
        if (lane == 0) {
            for (int s = 0; s < S; ++s) {
                tc_mbar_init(full_bar + 8 * s, 1);
                tc_mbar_init(empty_bar + 8 * s, 1);
            }
            for (int a = 0; a < A; ++a) {
                tc_mbar_init(tfull_bar + 8 * a, 1);
                tc_mbar_init(tempty_bar + 8 * a, kTcEpiWarps);
            }
            for (int b = 0; b < 2; ++b) {
                tc_mbar_init(qfull_bar + 8 * b, 1);
                tc_mbar_init(qempty_bar + 8 * b, 1);
                tc_mbar_init(tbfull_bar + 8 * b, 1);
                tc_mbar_init(tbfree_bar + 8 * b, kTcEpiWarps);
            }
            tc_mbar_init(mdone_bar, 1);
            *abort = 0;
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&smap)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&qmap)) : "memory");
        }
        // Tiles of request r's row sets: gblocks x TcReq(r).tiles.  Pass 1 counts
        // them all, pass 2 finds the request holding this CTA's first tile.
        constexpr int kB = 8;   // seq_lens loads in flight per lane
        auto req_tiles = [&](int64_t r) -> int64_t {
            return r < p.reqs ? static_cast<int64_t>(p.gblocks) * TcReq<QL, GB>(p, r).tiles : 0;
        };
        int64_t total = 0;
        for (int64_t r0 = 0; r0 < p.reqs; r0 += 32 * kB) {
            int64_t v[kB];
#pragma unroll
            for (int e = 0; e < kB; ++e)
                v[e] = req_tiles(r0 + e * 32 + lane);
#pragma unroll
            for (int e = 0; e < kB; ++e)
                total += v[e];
        }
        for (int o = 16; o; o >>= 1)
            total += __shfl_xor_sync(~0u, total, o);
        const int64_t lo = total * blockIdx.x / gridDim.x, hi = total * (blockIdx.x + 1) / gridDim.x;
        int64_t before = 0;     // tiles of the requests already passed
        bool found = false;
        for (int64_t r0 = 0; r0 < p.reqs && !found; r0 += 32) {
            const int64_t r = r0 + lane;
            const int64_t v = req_tiles(r);
            int64_t incl = v;
            for (int o = 1; o < 32; o <<= 1) {
                const int64_t x = __shfl_up_sync(~0u, incl, o);
                if (lane >= o)
                    incl += x;
            }
            const int64_t excl = before + incl - v;
            const bool here = v > 0 && excl <= lo && lo < excl + v;
            const unsigned m = __ballot_sync(~0u, here);
            if (here) {
                const int64_t per = v / p.gblocks;    // tiles of one row set of request r
                start[0] = r;
                start[1] = (lo - excl) / per;
                start[2] = (lo - excl) % per;
                start[3] = hi - lo;
            }
            found = m != 0;
            before += __shfl_sync(~0u, incl, 31);
        }
        if (!found && lane == 0) {   // an empty range
            start[0] = p.reqs;
            start[1] = start[2] = start[3] = 0;
        }
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(sbase + C::kTmemSlot),
                     "n"(C::kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sm + C::kTmemSlot);

    if (warp == 0) {
        // ---- producer.  The page ids of piece a's runs sit in tbuf[a & 1] (-1:
        // past the scored regions or no valid page), where the epilogue reads
        // them too; the next piece's are loaded into registers while this
        // piece's tiles are copied.
        constexpr int kPer = (C::kPieceRuns + 31) / 32;   // table entries per lane and piece
        int64_t pg[kPer];
        auto fetch = [&](const TcPiece<QL, GB> &pc) {
            const int32_t *trow = p.table + pc.req * p.bt_s0;
#pragma unroll
            for (int e = 0; e < kPer; ++e) {
                const int k = e * 32 + lane;
                const int j = pc.lo() + 8 * k;
                pg[e] = -2;                           // -2: no region to score here
                if (k < pc.nt * R && j < pc.rq.n_max) {
                    const int64_t col = static_cast<int64_t>(j) * kRegionTokens / p.block;
                    pg[e] = col < p.width ? trow[col] : -1;
                }
            }
        };
        TcCursor<QL, GB> cur(p, start);
        TcPiece<QL, GB> pc, nx;
        bool have = cur.next(p, pc);
        if (have)
            fetch(pc);
        int issued = 0;                               // tiles issued (stage ring position)
        bool stop = false;
        for (int a = 0; have && !stop; ++a) {
            const int b = a & 1;
            int32_t *tb = tbuf + b * C::kPieceRuns;
            if (a >= 2) {                             // the epilogue is done with piece a - 2's ids
                bool ok = true;
                if (lane == 0)
                    ok = tc_wait(tbfree_bar + 8 * b, ((a >> 1) - 1) & 1, p.wait_ns, abort);
                if (!__shfl_sync(~0u, ok, 0)) {
                    if (lane == 0) {
                        *abort = 1;
                        if (p.flags)
                            atomicOr(p.flags, SDA_FLAG_TIMEOUT);
                    }
                    break;
                }
            }
#pragma unroll
            for (int e = 0; e < kPer; ++e) {
                const int k = e * 32 + lane;
                if (k >= C::kPieceRuns)
                    continue;
                const bool ok = pg[e] >= 0 && pg[e] < p.pages;
                if (!ok && pg[e] != -2 && p.flags)
                    atomicOr(p.flags, SDA_FLAG_BOUNDS);
                tb[k] = ok ? static_cast<int32_t>(pg[e]) : -1;
            }
            __syncwarp();
            if (lane == 0)
                tc_mbar_arrive(tbfull_bar + 8 * b);
            const bool have_next = cur.next(p, nx);
            if (have_next)
                fetch(nx);                            // in flight during this piece's copies
            for (int t = 0; t < pc.nt; ++t) {
                const int s = issued % S;
                if (issued >= S) {
                    bool ok = true;
                    if (lane == 0)
                        ok = tc_wait(empty_bar + 8 * s, ((issued / S) - 1) & 1, p.wait_ns, abort);
                    if (!__shfl_sync(~0u, ok, 0)) {
                        if (lane == 0) {
                            *abort = 1;
                            if (p.flags)
                                atomicOr(p.flags, SDA_FLAG_TIMEOUT);
                        }
                        stop = true;
                        break;
                    }
                }
                const int page = lane < R ? tb[t * R + lane] : -1;
                const unsigned issue = __ballot_sync(~0u, page >= 0);
                const uint32_t fb = full_bar + 8 * s;
                if (lane == 0)
                    tc_mbar_expect_tx(fb, __popc(issue) * kBoxBytes);
                __syncwarp();
                if (page >= 0) {
                    const int j = pc.lo() + t * C::kRegions + 8 * lane;
                    tc_tma_5d(sbase + s * kTcTileBytes + lane * kBoxBytes, &smap, 0, j % p.per_page, 0, pc.gb0,
                              page, fb);
                }
                __syncwarp();
                if (lane == 0)
                    tc_mbar_arrive(fb);
                ++issued;
            }
            pc = nx;
            have = have_next;
        }
        // every copy this CTA started lands before the CTA can exit
        if (lane == 0)
            for (int k = issued > S ? issued - S : 0; k < issued; ++k)
                tc_wait(full_bar + 8 * (k % S), (k / S) & 1, kTcDrainNs);
    } else if (warp == 1) {
        // ---- MMA issue (one thread).  Query buffer a & 1 holds piece a's query
        // rows; the next piece's rows load into the other buffer while this
        // piece's tiles run.
        if (lane == 0) {
            const uint32_t q0 = sbase + C::kQ;
            auto load_q = [&](const TcPiece<QL, GB> &pc, int b) {
                const uint32_t dst = q0 + b * C::kQBuf;
                const int tok0 = static_cast<int>(pc.req * QL);
                tc_mbar_expect_tx(qfull_bar + 8 * b, 2 * kQBoxBytes);
                tc_tma_5d(dst, &qmap, 0, 0, 0, pc.gb0, tok0, qfull_bar + 8 * b);
                tc_tma_5d(dst + N * 128, &qmap, 0, 1, 0, pc.gb0, tok0, qfull_bar + 8 * b);
                tc_mbar_arrive(qfull_bar + 8 * b);
            };
            TcCursor<QL, GB> cur(p, start);
            TcPiece<QL, GB> pc, nx;
            bool have = cur.next(p, pc);
            int done = 0;               // tiles issued
            int q_loads = 0;            // query loads issued (piece a's load is number a)
            bool ok = true;
            if (have) {
                load_q(pc, 0);
                q_loads = 1;
            }
            for (int a = 0; have && ok; ++a) {
                const int b = a & 1;
                ok = tc_wait(qfull_bar + 8 * b, (a >> 1) & 1, p.wait_ns, abort);
                const bool have_next = cur.next(p, nx);
                if (ok && have_next) {
                    // buffer b ^ 1 was last read by piece a - 1's MMAs
                    if (a >= 1)
                        ok = tc_wait(qempty_bar + 8 * (b ^ 1), ((a - 1) >> 1) & 1, p.wait_ns, abort);
                    if (ok) {
                        load_q(nx, b ^ 1);
                        ++q_loads;
                    }
                }
                const uint32_t qb = q0 + b * C::kQBuf;
                for (int t = 0; t < pc.nt && ok; ++t, ++done) {
                    const int s = done % S, acc = done % A;
                    ok = tc_wait(full_bar + 8 * s, (done / S) & 1, p.wait_ns, abort);
                    if (ok && done >= A)
                        ok = tc_wait(tempty_bar + 8 * acc, ((done / A) - 1) & 1, p.wait_ns, abort);
                    if (!ok)
                        break;
                    tc_fence_after();
                    const uint32_t a0 = sbase + s * kTcTileBytes;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {   // K step of 32 bytes: half k / 4, offset 32 (k % 4)
                        const uint32_t ka = (k >> 2) * 1024 + (k & 3) * 32;
                        const uint32_t kb = (k >> 2) * (N * 128) + (k & 3) * 32;
                        tc_mma(tmem + acc * N, tc_desc_sw128(a0 + ka, 2048), tc_desc_sw128(qb + kb, 1024), kIdesc,
                               k > 0 ? 1u : 0u);
                    }
                    tc_commit(empty_bar + 8 * s);      // the stage is free once these MMAs have read it
                    tc_commit(tfull_bar + 8 * acc);    // the accumulator is ready
                }
                tc_commit(qempty_bar + 8 * b);         // query buffer b is free once they complete
                pc = nx;
                have = have_next;
            }
            if (!ok) {
                *abort = 1;
                if (p.flags)
                    atomicOr(p.flags, SDA_FLAG_TIMEOUT);
            }
            // Before the CTA releases its tensor memory and exits: every query load
            // it started has landed (loads into one buffer complete in order), and
            // every MMA it issued has completed.
            for (int l = q_loads > 2 ? q_loads - 2 : 0; l < q_loads; ++l)
                tc_wait(qfull_bar + 8 * (l & 1), (l >> 1) & 1, kTcDrainNs);
            tc_commit(mdone_bar);
            tc_wait(mdone_bar, 0, kTcDrainNs);
        }
        __syncwarp();
    } else {
        // ---- epilogue: 8 warps, two per tensor-memory lane quarter (warp % 4);
        // the first of each pair handles tokens [0, (QL + 1) / 2), the second
        // the rest.  Row m = 32 q + lane is run m / (8 GB), group m / 8 % GB,
        // slot m % 8.
        if ((warp - 2) < 4)
            tc_epilogue<QL, GB, 0, (QL + 1) / 2>(p, tmem, tbuf, start, tfull_bar, tempty_bar, tbfull_bar,
                                                 tbfree_bar, abort);
        else
            tc_epilogue<QL, GB, (QL + 1) / 2, QL>(p, tmem, tbuf, start, tfull_bar, tempty_bar, tbfull_bar,
                                                  tbfree_bar, abort);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(C::kTmemCols)
                     : "memory");
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

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn index_encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// The tensor-core variant when the pages fit its tiles: a page's summary
// slots (block / 8 of them) a multiple of 8 that divides the 128-region tile
// or is a multiple of it, and a whole number of pages in `summaries`.
// Returns SDA_ERR_UNSUPPORTED (and launches nothing) when it does not apply.
template <int QL, int GB>
cudaError_t launch_tc_kernel(const CUtensorMap &smap, const CUtensorMap &qmap, const IndexTcParams &tp,
                             int64_t grid, cudaStream_t stream)
{
    using C = TcCfg<QL, GB>;
    const void *kernel = reinterpret_cast<const void *>(sda_index_tc_kernel<QL, GB>);
    static std::mutex mu;
    static bool raised[256] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 0 || dev >= 256 || !raised[dev]) {
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kAlloc);
            if (e != cudaSuccess)
                return e;
            if (dev >= 0 && dev < 256)
                raised[dev] = true;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = C::kAlloc;
    cfg.stream = stream;
    CUtensorMap sm = smap, qm = qmap;
    IndexTcParams prm = tp;
    void *args[] = {&sm, &qm, &prm};
    return cudaLaunchKernelExC(&cfg, kernel, args);
}

// The tensor-core variant when the pages fit its tiles: a page's summary
// slots (block / 8 of them) a multiple of 8, and a whole number of pages in
// `summaries`.  Returns SDA_ERR_UNSUPPORTED (and launches nothing) when it
// does not apply.
sda_status launch_tc(const sda_tensor *query, const sda_tensor *summaries, const IndexParams &ip,
                     int query_len, int gblock, int64_t tokens, int64_t reqs, cudaStream_t stream)
{
    const int per_page = ip.block / kRegionTokens;
    if (ip.block % 64 != 0 || ip.n_slots % per_page != 0 || ip.n_cols < 1)
        return SDA_ERR_UNSUPPORTED;
    const int64_t pages = ip.n_slots / per_page;
    const int64_t groups = ip.groups;
    if (pages < 1 || pages > INT32_MAX || tokens > INT32_MAX)
        return SDA_ERR_UNSUPPORTED;
    EncodeTiledFn encode = index_encode_fn();
    if (!encode)
        return SDA_ERR_UNSUPPORTED;
    const cuuint32_t estride[5] = {1, 1, 1, 1, 1};
    CUtensorMap smap, qmap;
    // summaries as (128-byte K chunk, slot in page, K half, group, page): one box is
    // 8 slots x both halves x gblock groups of one page
    {
        const cuuint64_t gdim[5] = {128u, static_cast<cuuint64_t>(per_page), 2u, static_cast<cuuint64_t>(groups),
                                    static_cast<cuuint64_t>(pages)};
        const cuuint64_t gstride[4] = {static_cast<cuuint64_t>(ip.m_s0), 128u, static_cast<cuuint64_t>(kIdxDim),
                                       static_cast<cuuint64_t>(ip.m_s0) * static_cast<cuuint64_t>(per_page)};
        const cuuint32_t box[5] = {128u, 8u, 2u, static_cast<cuuint32_t>(gblock), 1u};
        if (encode(&smap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void *>(summaries->data), gdim, gstride,
                   box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return SDA_ERR_UNSUPPORTED;
    }
    // queries as (128-byte K chunk, K half, head, group, token): one box per K half
    // holds the query_len tokens' gblock groups' 8 heads as rows (token, group, head)
    {
        const cuuint64_t gdim[5] = {128u, 2u, static_cast<cuuint64_t>(kIdxHeads), static_cast<cuuint64_t>(groups),
                                    static_cast<cuuint64_t>(tokens)};
        const cuuint64_t gstride[4] = {128u, static_cast<cuuint64_t>(kIdxDim), static_cast<cuuint64_t>(ip.q_s1),
                                       static_cast<cuuint64_t>(ip.q_s0)};
        const cuuint32_t box[5] = {128u, 1u, static_cast<cuuint32_t>(kIdxHeads), static_cast<cuuint32_t>(gblock),
                                   static_cast<cuuint32_t>(query_len)};
        if (encode(&qmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void *>(query->data), gdim, gstride, box,
                   estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return SDA_ERR_UNSUPPORTED;
    }
    IndexTcParams tp;
    tp.weights = ip.weights;
    tp.w_s0 = ip.w_s0;
    tp.w_s1 = ip.w_s1;
    tp.table = ip.table;
    tp.bt_s0 = ip.bt_s0;
    tp.width = ip.width;
    tp.seq_lens = ip.seq_lens;
    tp.sl_s0 = ip.sl_s0;
    tp.scores = ip.scores;
    tp.sc_s0 = ip.sc_s0;
    tp.current = ip.current;
    tp.cur_s0 = ip.cur_s0;
    tp.lengths = ip.lengths;
    tp.len_s0 = ip.len_s0;
    tp.flags = ip.flags;
    tp.pages = pages;
    tp.wait_ns = sda_wait_limit_ns();
    tp.groups = ip.groups;
    tp.gblocks = ip.groups / gblock;
    tp.block = ip.block;
    tp.n_cols = ip.n_cols;
    tp.per_page = per_page;
    tp.reqs = reqs;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        return SDA_ERR_CUDA;
    // one CTA per SM, or fewer when there are fewer tiles than that (a row set has
    // at most ceil(n_cols / regions per tile) tiles); a CTA whose share of the
    // tiles is empty sets up and returns
    const int64_t regions = kTcM / 8 / gblock * 8;
    const int64_t max_tiles = reqs * tp.gblocks * ((ip.n_cols + regions - 1) / regions);
    const int64_t grid = std::min<int64_t>(max_tiles, static_cast<int64_t>(sms) * kTcCtasPerSm);
    if (grid < 1)
        return SDA_OK;
    using Fn = cudaError_t (*)(const CUtensorMap &, const CUtensorMap &, const IndexTcParams &, int64_t,
                               cudaStream_t);
    const Fn fns[kMaxQueryLen][3] = {
        {launch_tc_kernel<1, 1>, launch_tc_kernel<1, 2>, launch_tc_kernel<1, 4>},
        {launch_tc_kernel<2, 1>, launch_tc_kernel<2, 2>, launch_tc_kernel<2, 4>},
        {launch_tc_kernel<3, 1>, launch_tc_kernel<3, 2>, launch_tc_kernel<3, 4>},
        {launch_tc_kernel<4, 1>, launch_tc_kernel<4, 2>, launch_tc_kernel<4, 4>}};
    const int slot = gblock == 4 ? 2 : gblock - 1;
    return fns[query_len - 1][slot](smap, qmap, tp, grid, stream) == cudaSuccess ? SDA_OK : SDA_ERR_CUDA;
}

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
    // Pages of a multiple of 64 tokens take the tensor-core variant.
    {
        const sda_status st = launch_tc(query, summaries, prm, query_len, gblock, tokens, reqs,
                                        static_cast<cudaStream_t>(stream));
        if (st != SDA_ERR_UNSUPPORTED)
            return st;
    }
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
