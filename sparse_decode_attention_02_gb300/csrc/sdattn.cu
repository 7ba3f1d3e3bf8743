// GB300 (sm_103a) DSA sparse decode attention over a paged KV cache.
//
// Implements the operation of the vLLM API page
// "vllm.models.step5.nvidia.ops.sparse_decode_attention" (function
// `sparse_decode_attention`, helper `_gate`, policy `sparse_decode_splits`)
// behind the C ABI declared in include/sdattn.h.
//
// Design (one CTA per (row, split) unit; 5 warps):
//   * warp 4 (producer) compacts the row's live regions, splits them into a
//     contiguous chunk per split, resolves each region's pages through
//     block_table (one lane per piece, the next batch's table entries loading
//     meanwhile) and streams "pieces" (runs of P = min(RT, B, stage) tokens of
//     one page) into a 4-stage ring: the lanes holding a stage's pieces issue
//     one 5-D TMA box each (128-byte band chunks x P tokens x all bands of the
//     [pages, G, B, 384] cache, 128-byte swizzle);
//   * warps 0-3 (consumers) work in two pairs that take alternate stages, each
//     warp owning half of a stage's slots: QK^T for the 16-head x 192 query
//     tile with mma.sync m16n8k16 (heads are the M dimension), causal/validity
//     masking, online softmax in fp32, PV with mma.sync; FP8 bytes are
//     converted to fp16 in registers;
//   * the epilogue merges the warps' (max, sum, O) through shared memory and
//     either writes the gated bf16 output (one split) or the split's fp32
//     partial output and log-sum-exp for the combine kernel.
// Window mode walks the pieces of [pos - window + 1, pos] instead of regions;
// with token pairs one CTA serves two query tokens of a request (their
// overlapping windows streamed once, one warp pair per token; with a bf16
// cache the two warps of a token take alternate stages, all slots each).
// Every mbarrier wait is bounded; a wait that runs out raises a flag in the
// workspace header and the CTA winds down after its copies have landed.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "sdattn.h"

namespace {

constexpr int kDim = 192;
constexpr int kRow = 384;
constexpr int kMaxHeads = 16;
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxSplits = 64;
constexpr int kObufStride = 208;           // floats per head row of the epilogue buffer
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleSlack = 8.0f;      // log2 units a running max may lag the true max
constexpr size_t kHeaderBytes = 256;
constexpr uint64_t kDrainLimitNs = 1000000000ull;

// Diagnostic builds (compiled with SDA_TIMELINE) stamp %globaltimer at phase
// boundaries into a device buffer registered with sparse_decode_timeline_buffer:
// split CTA u writes entries u * 8 + k (k = 0 entry, 1 consumers released, 2
// first stage seen, 3 stage loop done, 4 output writes start, 5 done), combine
// CTA r entries kTimelineCombine + r * 2 + k (k = 0 entry, 1 past the wait on
// the split kernel).  The regular build compiles every stamp away.
constexpr unsigned long long kTimelineUnits = 1ull << 20;
constexpr unsigned long long kTimelineCombine = 8 * kTimelineUnits;
constexpr size_t kTimelineBytes = (8 + 2) * kTimelineUnits * sizeof(unsigned long long);
#ifdef SDA_TIMELINE
__device__ unsigned long long *g_sda_timeline = nullptr;
#define SDA_STAMP(cond, idx)                                                                       \
    do {                                                                                           \
        unsigned long long *tl_ = g_sda_timeline;                                                  \
        if ((cond) && tl_) {                                                                       \
            unsigned long long t_;                                                                 \
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                                  \
            tl_[idx] = t_;                                                                         \
        }                                                                                          \
    } while (0)
#else
#define SDA_STAMP(cond, idx) \
    do {                     \
    } while (0)
#endif


template <bool FP8>
struct Traits;
// A stage holds kSlots tokens as kBands column bands of 128 bytes per token.
// Two consumer warps share a stage (kWarpTokens slots each) and the two warp
// pairs take alternate stages, so a stage is released as soon as its pair is
// done with it.
template <>
struct Traits<true> {                      // FP8: 384 B per token; 4 stages of 64 tokens (24 KB)
    static constexpr int kBands = 3;
    static constexpr int kStages = 4;
    static constexpr int kElt = 1;
    static constexpr int kSlots = 64;
    static constexpr int kWarpTokens = 32;
    static constexpr int kBandBytes = kSlots * 128;
};
template <>
struct Traits<false> {                     // bf16: 768 B per token; 4 stages of 32 tokens (24 KB)
    static constexpr int kBands = 6;
    static constexpr int kStages = 4;
    static constexpr int kElt = 2;
    static constexpr int kSlots = 32;
    static constexpr int kWarpTokens = 16;
    static constexpr int kBandBytes = kSlots * 128;
};
constexpr int kWarpsPerStage = 2;
constexpr int kIdBatch = 8;               // region-id loads in flight per producer lane
constexpr int kPairs = kConsumerWarps / kWarpsPerStage;

constexpr int align_up(int x, int a)
{
    return (x + a - 1) / a * a;
}

// Shared memory of the split kernel, from a 1024-byte aligned base: the stage
// ring (1024-aligned stages for the 128-byte swizzle), mbarriers, stage
// headers, control words, per-warp softmax statistics, gate factors, the Q
// fragment array (16-byte vector accesses) and the row's live region list.
// With PAIR (two query tokens per CTA) the headers, gate factors and Q
// fragments come twice, one set per token.
template <bool FP8, bool PAIR = false>
struct Layout {
    static constexpr int kTokens = PAIR ? 2 : 1;
    static constexpr int kStageBytes = Traits<FP8>::kBands * Traits<FP8>::kBandBytes;
    static constexpr int kRing = Traits<FP8>::kStages * kStageBytes;
    static constexpr int kBarOff = kRing;
    static constexpr int kHdrOff = align_up(kBarOff + 16 * Traits<FP8>::kStages, 16);   // [token][stage]
    static constexpr int kCtlOff = align_up(kHdrOff + 8 * Traits<FP8>::kStages * kTokens, 16);
    static constexpr int kMlOff = kCtlOff + 64;
    static constexpr int kGammaOff = align_up(kMlOff + kConsumerWarps * kMaxHeads * 2 * 4, 16);
    static constexpr int kQOff = align_up(kGammaOff + kTokens * kMaxHeads * 4, 128);   // [token][12][32] x 16 B
    static constexpr int kQBytes = 12 * 32 * 16;
    static constexpr int kLiveOff = align_up(kQOff + kTokens * kQBytes, 16);
    static_assert(kStageBytes % 1024 == 0 && Traits<FP8>::kBandBytes % 1024 == 0, "swizzle atoms");
    static_assert(Traits<FP8>::kSlots == kWarpsPerStage * Traits<FP8>::kWarpTokens, "stage split");
    static_assert(kBarOff % 8 == 0 && kHdrOff % 8 == 0 && kQOff % 16 == 0, "alignment");
    static_assert(kRing >= kConsumerWarps * kMaxHeads * kObufStride * 4, "epilogue buffer");
    static size_t bytes(int num_regions) {
        return 1024 + kLiveOff + 4 * (size_t)((num_regions + 31) & ~31);
    }
};

struct Params {
    const uint16_t *query;
    int64_t q_s0, q_s1;
    const int32_t *regions;
    int64_t reg_s0;
    const int32_t *block_table;
    int64_t bt_s0;
    const int32_t *positions;
    int64_t pos_s0;
    const uint8_t *active;
    int64_t act_s0;
    uint16_t *output;
    int64_t o_s0, o_s1;
    const uint16_t *gate;
    int64_t g_s0, g_s1;
    const float *k_scale;
    const float *v_scale;
    float *partial;
    float *lse;
    unsigned int *flags;
    const int32_t *seq_lens;   // window mode: per-request lengths (positions derive from them)
    long long pages;
    unsigned long long wait_ns;
    float scale;
    int num_regions, table_cols;
    int rows, heads, groups, block, region_tokens, piece, query_len, splits;
    int clear_inactive;
    int window;                // > 0: sliding-window mode (no regions; every row active)
};

// ---------------------------------------------------------------------------
// PTX helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_init_fence()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
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

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for the phase of `bar` with the given parity; false after limit_ns.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (global_timer_ns() - t0 > limit_ns)
            return false;
    }
}

__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            int c3, int c4, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void consumer_bar()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                              uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

template <bool FP8>
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1)
{
    if constexpr (FP8) {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
            "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    } else {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
            "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
}

// Two E4M3 bytes (low byte -> low half) to two fp16 values, exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes)
{
    uint32_t r;
    const uint16_t v = static_cast<uint16_t>(two_bytes);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
    return r;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t sel)
{
    uint32_t r;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(r) : "r"(a), "r"(sel));
    return r;
}

template <bool FP8>
__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    uint32_t r;
    if constexpr (FP8)
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b)
{
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// `_gate`: sigmoid in fp32 (1 / (1 + exp(-g)) with a round-to-nearest
// division), rounded to bf16 and read back as fp32.
__device__ __forceinline__ float gate_factor(uint16_t g_bits)
{
    const float g = bf16_bits_to_float(g_bits);
    const float sig = __fdiv_rn(1.0f, 1.0f + expf(-g));
    return __bfloat162float(__float2bfloat16_rn(sig));
}

// FP8 path: the power-of-two exponent e by which a consumer warp scales its
// token's q before the fp16 MMA, from the per-warp maxima of the bf16 bit
// patterns (|q|) that the consumers left in ctl[4..7]: e puts the largest |q|
// in [2^14, 2^15) (14 - unbiased exponent, subnormals as the smallest
// exponent), clamped so that 2^e and 2^-e stay normal fp32 numbers; 0 for an
// all-zero q and on the bf16 path.
template <bool FP8, bool PAIR>
__device__ __forceinline__ int q_prescale_exp(const volatile int *ctl, int warp)
{
    if constexpr (!FP8) {
        return 0;
    } else {
        const int m = PAIR ? max(ctl[4 + (warp & 2)], ctl[5 + (warp & 2)])
                           : max(max(ctl[4], ctl[5]), max(ctl[6], ctl[7]));
        return m ? min(126, max(-126, 141 - max(1, m >> 7))) : 0;
    }
}

// Token slot of k-index n (0..7) inside an 8-slot group.  Pairs of fragment
// columns (2p, 2p+1) map to slots (p, p+4) so that the eight 16-byte K reads
// of one shared-memory phase hit eight different swizzled chunks.
__device__ __forceinline__ int rowmap(int n)
{
    return (n >> 1) | ((n & 1) << 2);
}

// A stage holds its pieces of P slots one after another, each stored as
// [band][row][128 bytes] (one TMA box), so the 8-slot tile starting at slot s
// (8 | P, 8 | s) sits at this byte offset and its bands are P * 128 bytes
// apart.  With P = slots per stage this is the plain [band][slot] layout.
// Tiles past the stage's last piece (P not dividing the stage) alias tile 0:
// their slots are never valid.
__device__ __forceinline__ uint32_t tile_offset(int s, int P, int pieces_per_stage, uint32_t piece_stride)
{
    const int k = s / P;
    return k < pieces_per_stage ? k * piece_stride + static_cast<uint32_t>(s - k * P) * 128u : 0u;
}

// O[16 heads x 192] += P[16 x 16 slots] V[16 slots x 192] for one warp.  V is
// read with ldmatrix.trans from the stage's V bands: lane `mi = lane / 8`
// addresses k-slots (mi & 1) * 8 + 0..7 of chunk (mi >> 1) of a chunk pair;
// `vrow` is this lane's slot row, `vsw` its swizzle phase.  MASKED zeroes the
// V values of invalid slots (vm0: k-slots 2t, 2t+1; vm1: 8+2t, 9+2t).
template <bool FP8, bool MASKED>
__device__ __forceinline__ void pv_accumulate(float (&o)[24][4], const uint32_t (&pa)[4], uint32_t vrow,
                                              uint32_t bstride, int mi, int vsw, uint32_t vm0, uint32_t vm1)
{
    if constexpr (FP8) {
        // 16-dim chunks cv = 0..11: V dims 0..63 sit in band 1 chunks 4..7,
        // dims 64..191 in band 2 chunks 0..7.  One chunk gives two n8 tiles:
        // even dims (tile 2*cv) and odd dims (tile 2*cv + 1).
#pragma unroll
        for (int c2 = 0; c2 < 6; ++c2) {
            const int cv = 2 * c2 + (mi >> 1);
            const int band = cv < 4 ? 1 : 2;
            const int ch = cv < 4 ? cv + 4 : cv - 4;
            uint32_t r0, r1, r2, r3;
            ldsm_x4_trans(vrow + band * bstride + ((ch ^ vsw) << 4), r0, r1, r2, r3);
            if constexpr (MASKED) {
                r0 &= vm0;
                r1 &= vm1;
                r2 &= vm0;
                r3 &= vm1;
            }
            const uint32_t x0 = prmt(r0, 0x3120u), x1 = prmt(r1, 0x3120u);
            const uint32_t x2 = prmt(r2, 0x3120u), x3 = prmt(r3, 0x3120u);
            mma16816<true>(o[4 * c2 + 0], pa, e4m3x2_to_f16x2(x0), e4m3x2_to_f16x2(x1));
            mma16816<true>(o[4 * c2 + 1], pa, e4m3x2_to_f16x2(x0 >> 16), e4m3x2_to_f16x2(x1 >> 16));
            mma16816<true>(o[4 * c2 + 2], pa, e4m3x2_to_f16x2(x2), e4m3x2_to_f16x2(x3));
            mma16816<true>(o[4 * c2 + 3], pa, e4m3x2_to_f16x2(x2 >> 16), e4m3x2_to_f16x2(x3 >> 16));
        }
    } else {
        // 8-dim chunks cv = 0..23 in bands 3..5; one n8 tile each.
#pragma unroll
        for (int c2 = 0; c2 < 12; ++c2) {
            const int cv = 2 * c2 + (mi >> 1);
            const int band = 3 + (cv >> 3);
            const int ch = cv & 7;
            uint32_t r0, r1, r2, r3;
            ldsm_x4_trans(vrow + band * bstride + ((ch ^ vsw) << 4), r0, r1, r2, r3);
            if constexpr (MASKED) {
                r0 &= vm0;
                r1 &= vm1;
                r2 &= vm0;
                r3 &= vm1;
            }
            mma16816<false>(o[2 * c2], pa, r0, r1);
            mma16816<false>(o[2 * c2 + 1], pa, r2, r3);
        }
    }
}

// ---------------------------------------------------------------------------
// Split kernel
// ---------------------------------------------------------------------------

// FULL: a piece fills a whole stage (P = slots per stage), so the stage
// layout is a compile-time [band][slot] one.  PAIR (window mode, even
// query_len): a CTA serves two consecutive query tokens of a request and
// group, whose windows are one token apart; the producer streams (its split's
// share of) their union once, each warp pair computes one token over every
// stage (bf16: its two warps on alternate stages) and writes that token's row
// (output, or partial and LSE).
template <bool FP8, bool WINDOW, bool FULL, bool PAIR>
__global__ void __launch_bounds__(kThreads, 2)
    sda_split_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ Params p)
{
    static_assert(!PAIR || WINDOW, "token pairs are a window-mode layout");
    using T = Traits<FP8>;
    using L = Layout<FP8, PAIR>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t full_bar = sbase + L::kBarOff;
    const uint32_t empty_bar = full_bar + 8 * T::kStages;
    uint64_t *hdr = reinterpret_cast<uint64_t *>(smem + L::kHdrOff);
    int *ctl = reinterpret_cast<int *>(smem + L::kCtlOff);
    float *ml = reinterpret_cast<float *>(smem + L::kMlOff);
    float *gam = reinterpret_cast<float *>(smem + L::kGammaOff);
    int *live = reinterpret_cast<int *>(smem + L::kLiveOff);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // this warp's Q fragment array (PAIR: its warp pair's token)
    const uint32_t qfrag = sbase + L::kQOff + (PAIR && warp < kConsumerWarps ? (warp >> 1) * L::kQBytes : 0);
    // CTA (u, split) = blockIdx.x; with PAIR, unit u serves rows (token 2k,
    // group g) and (token 2k + 1, g), u = k * G + g, and `row` is the first.
    const int unit = static_cast<int>(blockIdx.x / static_cast<unsigned>(p.splits));
    const int split = static_cast<int>(blockIdx.x % static_cast<unsigned>(p.splits));
    const int row = PAIR ? (unit / p.groups) * 2 * p.groups + unit % p.groups : unit;

    if (warp == kConsumerWarps) {          // the producer warp owns the pipeline barriers
        if (lane == 0) {
            for (int s = 0; s < T::kStages; ++s) {
                mbar_init(full_bar + 8 * s, 1);
                mbar_init(empty_bar + 8 * s, (PAIR && FP8) ? kConsumerWarps : kWarpsPerStage);
            }
            mbar_init_fence();
            prefetch_tmap(&tmap);
        }
        __syncwarp();
    }
    pdl_launch_dependents();
    pdl_wait();   // inputs may be written by the previous kernel on the stream
    SDA_STAMP(threadIdx.x == 0 && blockIdx.x < kTimelineUnits, blockIdx.x * 8ull + 0);

    // Sparse mode: the row's selected regions, its position and active flag.
    // Window mode: every row is active; token j = (row / G) % query_len of a
    // request sits at seq_lens[request] - query_len + j and sees the window
    // [max(0, pos - window + 1), pos], walked as pieces (regions of P tokens).
    constexpr bool windowed = WINDOW;
    bool act = true;
    if constexpr (!WINDOW)
        act = p.active[row * p.act_s0] != 0;

    const int g = lane >> 2;               // fragment row group
    const int t = lane & 3;                // thread in quad

    // Producer-only row state.
    int64_t req = 0, win_lo = 0;
    int pos = 0, P = 0, npr = 0, win_base = 0;
    int pos_a = 0;                             // PAIR: the first token's position
    int64_t lo_b = 0;                          // PAIR: the second token's first visible token
    if (warp == kConsumerWarps) {
        req = row / (p.groups * p.query_len);
        pos = windowed ? p.seq_lens[req] - p.query_len + (row / p.groups) % p.query_len
                       : p.positions[row * p.pos_s0];
        P = p.piece;
        npr = p.region_tokens / P;             // pieces per region (1 in window mode)
        win_lo = windowed ? max(0, pos - p.window + 1) : 0;   // first visible token
        win_base = static_cast<int>(win_lo / P);              // its piece index
        if (PAIR) {                            // stream the union [window start of token a, pos of b]
            pos_a = pos;
            pos = pos_a + 1;
            lo_b = max(0, pos - p.window + 1);
        }
    }

    if (warp == kConsumerWarps) {
        // ---- Producer: compact the live regions of this row, in stored order.
        int n_live = 0;
        if (windowed) {
            n_live = pos >= 0 ? pos / P - win_base + 1 : 0;
        } else {
            // read whatever `active` says (the loads overlap), then drop inactive rows
            // ids are loaded kIdBatch x 32 at a time so their latencies overlap
            const int32_t *reg = p.regions + static_cast<int64_t>(row) * p.reg_s0;
            for (int j0 = 0; j0 < p.num_regions; j0 += 32 * kIdBatch) {
                int ids[kIdBatch];
#pragma unroll
                for (int b = 0; b < kIdBatch; ++b) {
                    const int j = j0 + 32 * b + lane;
                    ids[b] = j < p.num_regions ? __ldg(reg + j) : -1;
                }
#pragma unroll
                for (int b = 0; b < kIdBatch; ++b) {
                    const int id = ids[b];
                    if (act && id < -1)
                        atomicOr(p.flags, SDA_FLAG_BOUNDS);
                    const bool ok = act && id >= 0 && static_cast<int64_t>(id) * p.region_tokens <= pos;
                    const unsigned m = __ballot_sync(~0u, ok);
                    if (ok)
                        live[n_live + __popc(m & ((1u << lane) - 1u))] = id;
                    n_live += __popc(m);
                }
            }
        }
        __syncwarp();
        const int lo = static_cast<int>(static_cast<int64_t>(split) * n_live / p.splits);
        const int hi = static_cast<int>(static_cast<int64_t>(split + 1) * n_live / p.splits);
        long long pieces = 0;
        for (int i = lo + lane; i < hi; i += 32) {
            const int64_t first = static_cast<int64_t>(windowed ? win_base + i : live[i]) * p.region_tokens;
            pieces += min(static_cast<int64_t>(npr), (pos - first) / P + 1);
        }
        for (int o = 16; o; o >>= 1)
            pieces += __shfl_xor_sync(~0u, pieces, o);
        if (lane == 0) {
            const int per_stage = T::kSlots / P;   // P need not divide the stage
            ctl[0] = static_cast<int>((pieces + per_stage - 1) / per_stage);
            ctl[1] = lo;
            ctl[2] = hi;
        }
        __syncwarp();
        // Release the consumers (barriers, stage count) without waiting for
        // their Q fragments: the producer starts streaming right away.
        asm volatile("bar.arrive 2, %0;" ::"n"(kThreads) : "memory");
        SDA_STAMP(lane == 0 && blockIdx.x < kTimelineUnits, blockIdx.x * 8ull + 1);
    } else {
        // ---- Consumers: Q A-fragments into shared memory, in fragment order
        // ([k-step][lane] x 4 words).  K-step kk of thread t covers the four
        // dims d0..d0+3 that its K loads deliver (see the QK loop below).
        const int qrow = PAIR ? row + (warp >> 1) * p.groups : row;   // PAIR: the warp pair's token
        const uint16_t *q0 = p.query + static_cast<int64_t>(qrow) * p.q_s0;
        const int m0 = g, m1 = g + 8;
        const int kk0 = PAIR ? (warp & 1) : warp;
        constexpr int kKStride = PAIR ? 2 : kConsumerWarps;
        auto dim0 = [&](int kk) {
            if constexpr (FP8)
                return 64 * (kk >> 2) + 16 * t + 4 * (kk & 3);
            else
                return 64 * (kk >> 2) + 32 * ((kk >> 1) & 1) + 8 * t + 4 * (kk & 1);
        };
        auto q_bits = [&](int m, int d) -> uint32_t {
            return act && m < p.heads ? q0[static_cast<int64_t>(m) * p.q_s1 + d] : 0u;
        };
        if constexpr (FP8) {
            // The fp16 MMA takes q in fp16, whose range is far narrower than
            // bf16's.  Scale the row's q by 2^e so that its largest |q| lands
            // in [2^14, 2^15): every bf16 value within 2^31 of that maximum is
            // then exact in fp16, and 2^-e is folded back into the logit
            // scale, so the logits are those of the unscaled q up to fp32
            // rounding.  The maximum runs over all of the token's heads and
            // dims (this warp's k-steps, then the warps holding the token).
            uint32_t mx = 0;
#pragma unroll
            for (int kk = kk0; kk < 12; kk += kKStride) {
                const int d0 = dim0(kk);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    mx = max(mx, max(q_bits(m0, d0 + e), q_bits(m1, d0 + e)) & 0x7FFFu);
            }
            mx = __reduce_max_sync(~0u, mx);
            if (lane == 0)
                ctl[4 + warp] = static_cast<int>(mx);
            consumer_bar();
        }
        const float qs = __int_as_float((127 + q_prescale_exp<FP8, PAIR>(ctl, warp)) << 23);   // exact
#pragma unroll
        for (int kk = kk0; kk < 12; kk += kKStride) {
            const int d0 = dim0(kk);
            float a[2][4];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    a[r][e] = bf16_bits_to_float(static_cast<uint16_t>(q_bits(r ? m1 : m0, d0 + e))) * qs;
            }
            const uint32_t addr = qfrag + (kk * 32 + lane) * 16;
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                         "r"(pack2<FP8>(a[0][0], a[0][1])), "r"(pack2<FP8>(a[1][0], a[1][1])),
                         "r"(pack2<FP8>(a[0][2], a[0][3])), "r"(pack2<FP8>(a[1][2], a[1][3]))
                         : "memory");
        }
    }
    int n_st = 0;
    if (warp != kConsumerWarps) {           // wait for the producer's arrive and each other's Q stores
        asm volatile("bar.sync 2, %0;" ::"n"(kThreads) : "memory");
        n_st = ctl[0];
    }

    if (warp == kConsumerWarps) {
        // ---- Producer: stream pieces into the stage ring.
        const int lo = ctl[1], hi = ctl[2];
        const int grp = row % p.groups;
        const int32_t *bt = p.block_table + req * p.bt_s0;
        const int pps = T::kSlots / P;
        const uint32_t piece_bytes = static_cast<uint32_t>(P) * kRow * T::kElt;   // = one box
        int stage = 0, fill = 0, issued = 0;
        uint32_t phase = 0;
        uint64_t mask = 0, mask_a = 0;         // PAIR: mask is the second token's, mask_a the first's
        bool aborted = false;
        // Candidate pieces c = 0, 1, ... are (live region lo + c / npr, piece
        // c % npr); the visible ones fill the stages densely, in that order.
        // Each batch of 32 candidates is resolved one per lane, and the lanes
        // holding the pieces of a stage issue their copies together.
        const int n_cand = (hi - lo) * npr;
        // The next batch's table entries are loaded while this batch issues.
        bool nx_have = false, nx_col_ok = false;
        int nx_page = -1, nx_off = 0;
        int64_t nx_t0 = 0;
        auto fetch = [&](int b) {
            const int c = b + lane;
            nx_have = c < n_cand;
            const int i = lo + (nx_have ? c / npr : 0);
            const int j = nx_have ? c % npr : 0;
            const int id = nx_have ? (windowed ? win_base + i : live[i]) : 0;
            nx_t0 = static_cast<int64_t>(id) * p.region_tokens + static_cast<int64_t>(j) * P;
            nx_have = nx_have && nx_t0 <= pos;
            const int64_t col = nx_t0 / p.block;
            nx_off = static_cast<int>(nx_t0 - col * p.block);
            nx_col_ok = col < p.table_cols;
            nx_page = nx_have && nx_col_ok ? bt[col] : -1;
        };
        fetch(0);
        for (int base = 0; base < n_cand && !aborted; base += 32) {
            const bool have = nx_have;
            const int off = nx_off;
            const int64_t t0 = nx_t0;
            int page = nx_page;
            if (have && (!nx_col_ok || page < 0 || page >= p.pages)) {
                atomicOr(p.flags, SDA_FLAG_BOUNDS);
                page = -1;
            }
            if (base + 32 < n_cand)
                fetch(base + 32);
            // valid slots of the piece: [skip, nv) (skip > 0 only for a window's first piece)
            // valid slots of the piece for a token seeing [lo, hi]: [lo - t0, hi - t0 + 1) within [0, P)
            auto slot_bits = [&](int64_t lo, int64_t hi) -> uint64_t {
                const int64_t nv = have ? min(static_cast<int64_t>(P), max(static_cast<int64_t>(0), hi - t0 + 1)) : 0;
                const int64_t skip = have ? max(static_cast<int64_t>(0), lo - t0) : 0;
                const uint64_t upto = nv >= 64 ? ~0ull : ((1ull << nv) - 1ull);
                const uint64_t below = skip >= 64 ? ~0ull : ((1ull << skip) - 1ull);
                return upto & ~below;
            };
            const uint64_t pbits = slot_bits(PAIR ? lo_b : win_lo, pos);
            const uint64_t pbits_a = PAIR ? slot_bits(win_lo, pos_a) : 0ull;
            const unsigned hv = __ballot_sync(~0u, have);
            const int rank = __popc(hv & ((1u << lane) - 1u));
            const int nh = __popc(hv);
            for (int done = 0; done < nh;) {
                if (fill == 0 && issued >= T::kStages) {
                    if (lane == 0 && !mbar_wait(empty_bar + 8 * stage, phase ^ 1u, p.wait_ns)) {
                        atomicOr(p.flags, SDA_FLAG_TIMEOUT);
                        aborted = true;
                    }
                    aborted = __shfl_sync(~0u, aborted, 0);
                    if (aborted)
                        break;
                }
                const int take = min(pps - fill, nh - done);
                const bool mine = have && rank >= done && rank < done + take;
                const bool copy = mine && page >= 0;
                const unsigned cb = __ballot_sync(~0u, copy);
                const uint32_t fb = full_bar + 8 * stage;
                if (lane == 0 && cb)
                    mbar_expect_tx(fb, __popc(cb) * piece_bytes);
                __syncwarp();
                uint64_t mbits = 0, mbits_a = 0;
                if (copy) {
                    const int slot = fill + rank - done;
                    tma_load_5d(sbase + stage * L::kStageBytes + slot * piece_bytes, &tmap, 0, off, 0, grp,
                                page, fb);
                    mbits = pbits << (slot * P);
                    mbits_a = pbits_a << (slot * P);
                }
                const unsigned lo32 = __reduce_or_sync(~0u, static_cast<unsigned>(mbits));
                const unsigned hi32 = __reduce_or_sync(~0u, static_cast<unsigned>(mbits >> 32));
                mask |= (static_cast<uint64_t>(hi32) << 32) | lo32;
                if constexpr (PAIR) {
                    const unsigned alo = __reduce_or_sync(~0u, static_cast<unsigned>(mbits_a));
                    const unsigned ahi = __reduce_or_sync(~0u, static_cast<unsigned>(mbits_a >> 32));
                    mask_a |= (static_cast<uint64_t>(ahi) << 32) | alo;
                }
                fill += take;
                done += take;
                if (fill == pps) {
                    if (lane == 0) {
                        hdr[stage] = PAIR ? mask_a : mask;
                        if (PAIR)
                            hdr[T::kStages + stage] = mask;
                        mbar_arrive(fb);
                    }
                    ++issued;
                    fill = 0;
                    mask = 0;
                    mask_a = 0;
                    if (++stage == T::kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
        if (lane == 0) {
            if (fill > 0) {   // commit the last, partly filled stage (also after an abort)
                hdr[stage] = PAIR ? mask_a : mask;
                if (PAIR)
                    hdr[T::kStages + stage] = mask;
                mbar_arrive(full_bar + 8 * stage);
                ++issued;
            }
            // Let every copy this CTA started land before the consumers reuse
            // the ring for the epilogue and before any thread can exit.
            bool drained = true;
            for (int k = issued > T::kStages ? issued - T::kStages : 0; k < issued; ++k)
                drained = mbar_wait(full_bar + 8 * (k % T::kStages), static_cast<uint32_t>(k / T::kStages) & 1u,
                                    kDrainLimitNs) && drained;
            if (!drained)
                atomicOr(p.flags, SDA_FLAG_TIMEOUT);
            ctl[3] = drained ? 0 : 1;
        }
        __syncwarp();
        asm volatile("bar.arrive 3, %0;" ::"n"(kThreads) : "memory");   // ring drained (or given up)
        return;
    }

    // ---- Consumers.
    const float kfold = FP8 ? __ldg(p.k_scale) : 1.0f;
    const float vfold = FP8 ? __ldg(p.v_scale) : 1.0f;
    // Logit scale in log2 units.  FP8: with the q prescale undone (exact); it
    // passes through shared memory, which keeps the FP8 variants free of
    // register spills.
    float sl2 = p.scale * kLog2e * kfold;
    float *sl2_smem = reinterpret_cast<float *>(ctl + 8 + warp);
    if constexpr (FP8) {
        if (lane == 0)
            *sl2_smem = sl2 * __int_as_float((127 - q_prescale_exp<FP8, PAIR>(ctl, warp)) << 23);
        __syncwarp();
        sl2 = *sl2_smem;
    }

    float o[24][4];
#pragma unroll
    for (int n = 0; n < 24; ++n)
        o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.0f;
    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.0f, 0.0f};

    // This warp's pair takes stages pair, pair + 2, ...; inside a stage it owns
    // slots [slot0, slot0 + WT): NT token tiles of 8 for QK^T and KS k-steps
    // of 16 for PV.  PAIR: warps 2k and 2k + 1 serve token k; with FP8 both
    // take every stage (half its slots each), with bf16 (ALT) they take
    // alternate stages, all 32 slots each: four independent score tiles per
    // warp instead of two, and two arrivals per stage instead of four.
    constexpr bool ALT = PAIR && !FP8;
    constexpr int WT = ALT ? T::kSlots : T::kWarpTokens;
    constexpr int NT = WT / 8;
    constexpr int KS = WT / 16;
    const int pair = ALT ? (warp & 1) : PAIR ? 0 : warp / kWarpsPerStage;
    const uint64_t *my_hdr = hdr + (PAIR ? (warp >> 1) * T::kStages : 0);
    const int slot0 = ALT ? 0 : (warp % kWarpsPerStage) * T::kWarpTokens;
    constexpr uint64_t kWarpMask = (WT >= 64) ? ~0ull : ((1ull << WT) - 1ull);

    // Per-lane part of the V ldmatrix addresses: matrix mi = lane / 8 covers
    // k-slots (mi & 1) * 8 + 0..7 of chunk (mi >> 1) of the chunk pair.
    const int mi = lane >> 3;
    const int vk = (mi & 1) * 8 + (lane & 7);
    const int vsw = rowmap(vk & 7);        // swizzle phase of this lane's V rows
    const int sw = rowmap(g);              // swizzle phase of this lane's K rows
    // Stage offsets of this warp's K tile rows and V k-step rows, and the band stride.
    const int piece_c = FULL ? T::kSlots : p.piece;
    const int pps_c = T::kSlots / piece_c;
    const uint32_t bstride = static_cast<uint32_t>(piece_c) * 128u;
    const uint32_t pstride = bstride * T::kBands;
    uint32_t krow[NT], vrow_off[KS];
#pragma unroll
    for (int i = 0; i < NT; ++i)
        krow[i] = (FULL ? (slot0 + 8 * i) * 128u : tile_offset(slot0 + 8 * i, piece_c, pps_c, pstride)) +
                  sw * 128u;
#pragma unroll
    for (int k2 = 0; k2 < KS; ++k2)
        vrow_off[k2] = (FULL ? (slot0 + 16 * k2 + (vk & 8)) * 128u
                             : tile_offset(slot0 + 16 * k2 + (vk & 8), piece_c, pps_c, pstride)) +
                       vsw * 128u;

    for (int st = pair; st < n_st; st += ALT ? 2 : PAIR ? 1 : kPairs) {
        const int s = st % T::kStages;
        const uint32_t par = static_cast<uint32_t>(st / T::kStages) & 1u;
        const bool ok = mbar_wait(full_bar + 8 * s, par, p.wait_ns);
        SDA_STAMP(st == pair && warp == 0 && lane == 0 && blockIdx.x < kTimelineUnits, blockIdx.x * 8ull + 2);
        if (!__all_sync(~0u, ok)) {
            if (lane == 0)
                atomicOr(p.flags, SDA_FLAG_TIMEOUT);
            break;
        }
        const uint32_t wm = static_cast<uint32_t>((my_hdr[s] >> slot0) & kWarpMask);
        const uint32_t stage_base = sbase + s * L::kStageBytes;
        if (wm) {
            // ---- S = Q K^T for this warp's slots: tile i, column g is slot
            // slot0 + 8i + rowmap(g).
            float sc[NT][4];
#pragma unroll
            for (int i = 0; i < NT; ++i)
                sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.0f;
            if constexpr (FP8) {
                // thread t: band 0 chunks t and t+4, band 1 chunk t (16 dims each);
                // tiles in pairs to bound the live K words.
#pragma unroll
                for (int i0 = 0; i0 < NT; i0 += 2) {
#pragma unroll
                    for (int c = 0; c < 3; ++c) {
                        const int band = c == 2 ? 1 : 0;
                        const int ch = c == 1 ? t + 4 : t;
                        const uint32_t off = band * bstride + ((ch ^ sw) << 4);
                        const uint4 ka = lds128(stage_base + krow[i0] + off);
                        const uint4 kb = lds128(stage_base + krow[i0 + 1] + off);
                        const uint32_t wa[4] = {ka.x, ka.y, ka.z, ka.w};
                        const uint32_t wb[4] = {kb.x, kb.y, kb.z, kb.w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint4 qv = lds128(qfrag + ((4 * c + j) * 32 + lane) * 16);
                            const uint32_t qf[4] = {qv.x, qv.y, qv.z, qv.w};
                            mma16816<true>(sc[i0], qf, e4m3x2_to_f16x2(wa[j]), e4m3x2_to_f16x2(wa[j] >> 16));
                            mma16816<true>(sc[i0 + 1], qf, e4m3x2_to_f16x2(wb[j]), e4m3x2_to_f16x2(wb[j] >> 16));
                        }
                    }
                }
            } else {
                // thread t: bands 0-2, chunks t and t+4 (8 dims each, two k-steps)
#pragma unroll
                for (int j = 0; j < 6; ++j) {
                    const int band = j >> 1;
                    const int ch = (j & 1) * 4 + t;
                    const uint32_t off = band * bstride + ((ch ^ sw) << 4);
                    uint4 kv[NT];
#pragma unroll
                    for (int i = 0; i < NT; ++i)
                        kv[i] = lds128(stage_base + krow[i] + off);
                    const uint4 qa = lds128(qfrag + ((2 * j) * 32 + lane) * 16);
                    const uint4 qb = lds128(qfrag + ((2 * j + 1) * 32 + lane) * 16);
                    const uint32_t qfa[4] = {qa.x, qa.y, qa.z, qa.w};
                    const uint32_t qfb[4] = {qb.x, qb.y, qb.z, qb.w};
#pragma unroll
                    for (int i = 0; i < NT; ++i)
                        mma16816<false>(sc[i], qfa, kv[i].x, kv[i].y);
#pragma unroll
                    for (int i = 0; i < NT; ++i)
                        mma16816<false>(sc[i], qfb, kv[i].z, kv[i].w);
                }
            }

            // ---- Mask, online softmax.  In tile i, c0/c2 are slot 8i+t and
            // c1/c3 slot 8i+t+4 (relative to slot0).
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int i = 0; i < NT; ++i) {
                const bool v0 = (wm >> (8 * i + t)) & 1u;
                const bool v1 = (wm >> (8 * i + t + 4)) & 1u;
                sc[i][0] = v0 ? sc[i][0] * sl2 : -INFINITY;
                sc[i][1] = v1 ? sc[i][1] * sl2 : -INFINITY;
                sc[i][2] = v0 ? sc[i][2] * sl2 : -INFINITY;
                sc[i][3] = v1 ? sc[i][3] * sl2 : -INFINITY;
                mx0 = fmaxf(mx0, fmaxf(sc[i][0], sc[i][1]));
                mx1 = fmaxf(mx1, fmaxf(sc[i][2], sc[i][3]));
            }
            mx0 = fmaxf(mx0, __shfl_xor_sync(~0u, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(~0u, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(~0u, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(~0u, mx1, 2));
            const bool need = mx0 > m_run[0] + kRescaleSlack || mx1 > m_run[1] + kRescaleSlack;
            if (__any_sync(~0u, need)) {
                const float n0 = fmaxf(m_run[0], mx0), n1 = fmaxf(m_run[1], mx1);
                const float a0 = n0 == -INFINITY ? 1.0f : fast_exp2(m_run[0] - n0);
                const float a1 = n1 == -INFINITY ? 1.0f : fast_exp2(m_run[1] - n1);
                m_run[0] = n0;
                m_run[1] = n1;
                l_run[0] *= a0;
                l_run[1] *= a1;
#pragma unroll
                for (int n = 0; n < 24; ++n) {
                    o[n][0] *= a0;
                    o[n][1] *= a0;
                    o[n][2] *= a1;
                    o[n][3] *= a1;
                }
            }
            const float r0 = m_run[0] == -INFINITY ? 0.0f : m_run[0];
            const float r1 = m_run[1] == -INFINITY ? 0.0f : m_run[1];
            uint32_t pa[KS][4];
#pragma unroll
            for (int k2 = 0; k2 < KS; ++k2) {
                float pr[2][4];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int i = 2 * k2 + h;
                    pr[h][0] = fast_exp2(sc[i][0] - r0);   // -inf scores give 0
                    pr[h][1] = fast_exp2(sc[i][1] - r0);
                    pr[h][2] = fast_exp2(sc[i][2] - r1);
                    pr[h][3] = fast_exp2(sc[i][3] - r1);
                }
                l_run[0] += (pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]);
                l_run[1] += (pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]);
                pa[k2][0] = pack2<FP8>(pr[0][0], pr[0][1]);
                pa[k2][1] = pack2<FP8>(pr[0][2], pr[0][3]);
                pa[k2][2] = pack2<FP8>(pr[1][0], pr[1][1]);
                pa[k2][3] = pack2<FP8>(pr[1][2], pr[1][3]);
            }

            // ---- O += P V, one 16-slot k-step at a time.  Invalid slots' V may
            // hold anything (even NaN): zero them when a k-step is not all valid.
#pragma unroll
            for (int k2 = 0; k2 < KS; ++k2) {
                const uint32_t km = (wm >> (16 * k2)) & 0xFFFFu;
                const uint32_t vrow = stage_base + vrow_off[k2];
                if (km == 0xFFFFu) {
                    pv_accumulate<FP8, false>(o, pa[k2], vrow, bstride, mi, vsw, 0u, 0u);
                } else if (km) {
                    const uint32_t vm0 = (((km >> t) & 1u) ? 0x0000FFFFu : 0u) |
                                         (((km >> (t + 4)) & 1u) ? 0xFFFF0000u : 0u);
                    const uint32_t vm1 = (((km >> (t + 8)) & 1u) ? 0x0000FFFFu : 0u) |
                                         (((km >> (t + 12)) & 1u) ? 0xFFFF0000u : 0u);
                    pv_accumulate<FP8, true>(o, pa[k2], vrow, bstride, mi, vsw, vm0, vm1);
                }
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(empty_bar + 8 * s);
    }

    SDA_STAMP(threadIdx.x == 0 && blockIdx.x < kTimelineUnits, blockIdx.x * 8ull + 3);
    // ---- Epilogue: merge the four warps.
    float l0 = l_run[0], l1 = l_run[1];
    l0 += __shfl_xor_sync(~0u, l0, 1);
    l0 += __shfl_xor_sync(~0u, l0, 2);
    l1 += __shfl_xor_sync(~0u, l1, 1);
    l1 += __shfl_xor_sync(~0u, l1, 2);
    if (t == 0) {
        ml[(warp * kMaxHeads + g) * 2 + 0] = m_run[0];
        ml[(warp * kMaxHeads + g) * 2 + 1] = l0;
        ml[(warp * kMaxHeads + g + 8) * 2 + 0] = m_run[1];
        ml[(warp * kMaxHeads + g + 8) * 2 + 1] = l1;
    }
    const int ctid = threadIdx.x;          // 0..127 among consumers
    const int64_t tok = row / p.groups;
    const int grp = row % p.groups;
    if (ctid < L::kTokens * p.heads) {     // gam[token k][head h], token k = row's token + k
        const int k = ctid / p.heads, h = ctid - k * p.heads;
        gam[k * kMaxHeads + h] =
            p.gate ? gate_factor(p.gate[(tok + k) * p.g_s0 + static_cast<int64_t>(grp * p.heads + h) * p.g_s1])
                   : 1.0f;
    }
    // Every consumer's statistics are in shared memory, and the producer has
    // seen every copy it issued land (after a timed-out wait some may still
    // have been in flight), so the ring is free for the epilogue buffer.  If
    // the producer's drain itself ran out, the ring may still receive bytes:
    // the row is already flagged SDA_FLAG_TIMEOUT, and nothing more is written.
    asm volatile("bar.sync 3, %0;" ::"n"(kThreads) : "memory");
    if (ctl[3])
        return;

    float fac[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int h = g + 8 * r;
        // the warps holding this token: all four, or (PAIR) this warp's pair
        constexpr int kMerge = PAIR ? 2 : kConsumerWarps;
        const int w0 = PAIR ? (warp & 2) : 0;
        float M = -INFINITY;
#pragma unroll
        for (int w = w0; w < w0 + kMerge; ++w)
            M = fmaxf(M, ml[(w * kMaxHeads + h) * 2]);
        float Ls = 0.0f;
#pragma unroll
        for (int w = w0; w < w0 + kMerge; ++w) {
            const float mw = ml[(w * kMaxHeads + h) * 2];
            if (mw != -INFINITY)
                Ls += ml[(w * kMaxHeads + h) * 2 + 1] * fast_exp2(mw - M);
        }
        const float mine = m_run[r];
        fac[r] = (Ls > 0.0f && mine != -INFINITY) ? fast_exp2(mine - M) / Ls : 0.0f;
        if (p.splits > 1 && warp == w0 && t == 0 && h < p.heads && act)   // PAIR: pair k is row + k G
            p.lse[(static_cast<int64_t>(row + (PAIR ? (warp >> 1) * p.groups : 0)) * p.splits + split) *
                      p.heads + h] = Ls > 0.0f ? (M + log2f(Ls)) * kLn2 : -INFINITY;
    }

    // Scaled per-warp outputs into the (now idle) stage ring.
    float *obuf = reinterpret_cast<float *>(smem);
    float *ob0 = obuf + (warp * kMaxHeads + g) * kObufStride;
    float *ob1 = obuf + (warp * kMaxHeads + g + 8) * kObufStride;
    if constexpr (FP8) {
#pragma unroll
        for (int cv = 0; cv < 12; ++cv) {
            const int d = 16 * cv + 4 * t;
            *reinterpret_cast<float4 *>(ob0 + d) =
                make_float4(o[2 * cv][0] * fac[0], o[2 * cv + 1][0] * fac[0], o[2 * cv][1] * fac[0],
                            o[2 * cv + 1][1] * fac[0]);
            *reinterpret_cast<float4 *>(ob1 + d) =
                make_float4(o[2 * cv][2] * fac[1], o[2 * cv + 1][2] * fac[1], o[2 * cv][3] * fac[1],
                            o[2 * cv + 1][3] * fac[1]);
        }
    } else {
#pragma unroll
        for (int n = 0; n < 24; ++n) {
            const int d = 8 * n + 2 * t;
            *reinterpret_cast<float2 *>(ob0 + d) = make_float2(o[n][0] * fac[0], o[n][1] * fac[0]);
            *reinterpret_cast<float2 *>(ob1 + d) = make_float2(o[n][2] * fac[1], o[n][3] * fac[1]);
        }
    }
    consumer_bar();

    SDA_STAMP(threadIdx.x == 0 && blockIdx.x < kTimelineUnits, blockIdx.x * 8ull + 4);
    const int total = p.heads * kDim;
    if constexpr (PAIR) {                  // token k's rows: warps 2k and 2k + 1
        for (int e = ctid; e < 2 * total; e += kConsumerWarps * 32) {
            const int k = e >= total ? 1 : 0;
            const int r = e - k * total;
            const int h = r / kDim, d = r - h * kDim;
            const float v = (obuf[((2 * k) * kMaxHeads + h) * kObufStride + d] +
                             obuf[((2 * k + 1) * kMaxHeads + h) * kObufStride + d]) * vfold;
            const int64_t orow = row + k * p.groups;
            if (p.splits == 1) {
                uint16_t *out = p.output + orow * p.o_s0;
                out[static_cast<int64_t>(h) * p.o_s1 + d] =
                    __bfloat16_as_ushort(__float2bfloat16_rn(v * gam[k * kMaxHeads + h]));
            } else {                       // the combine kernel applies the gate
                p.partial[(orow * p.splits + split) * p.heads * kDim + r] = v;
            }
        }
    } else if (p.splits == 1) {
        if (!act && !p.clear_inactive)
            return;
        uint16_t *out = p.output + static_cast<int64_t>(row) * p.o_s0;
        for (int e = ctid; e < total; e += kConsumerWarps * 32) {
            const int h = e / kDim, d = e - h * kDim;
            float v = 0.0f;
            if (act) {
                v = obuf[h * kObufStride + d] + obuf[(kMaxHeads + h) * kObufStride + d] +
                    obuf[(2 * kMaxHeads + h) * kObufStride + d] + obuf[(3 * kMaxHeads + h) * kObufStride + d];
                v = v * vfold * gam[h];
            }
            out[static_cast<int64_t>(h) * p.o_s1 + d] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
        }
    } else if (act) {
        float *dst = p.partial + (static_cast<int64_t>(row) * p.splits + split) * p.heads * kDim;
        for (int e = ctid; e < total; e += kConsumerWarps * 32) {
            const int h = e / kDim, d = e - h * kDim;
            const float v = obuf[h * kObufStride + d] + obuf[(kMaxHeads + h) * kObufStride + d] +
                            obuf[(2 * kMaxHeads + h) * kObufStride + d] +
                            obuf[(3 * kMaxHeads + h) * kObufStride + d];
            dst[e] = v * vfold;
        }
    }
    SDA_STAMP(threadIdx.x == 0 && blockIdx.x < kTimelineUnits, blockIdx.x * 8ull + 5);
}

// ---------------------------------------------------------------------------
// Combine kernel: one CTA per row, one thread per (head, 4 dims).  Merges the
// splits through their LSEs (weights exp(lse_s - max), all -inf -> zeros),
// applies the gate and clears inactive rows.
// ---------------------------------------------------------------------------

constexpr int kCombineThreads = kMaxHeads * (kDim / 4);   // 768

__global__ void __launch_bounds__(kCombineThreads) sda_combine_kernel(const __grid_constant__ Params p)
{
    SDA_STAMP(threadIdx.x == 0 && blockIdx.x < kTimelineUnits, kTimelineCombine + blockIdx.x * 2ull);
    const int row = blockIdx.x;
    const int item = threadIdx.x;
    const bool mine = item < p.heads * (kDim / 4);
    const int h = mine ? item / (kDim / 4) : 0;
    const int d = 4 * (item - h * (kDim / 4));
    // Inputs the split kernel does not write (activity, gate) are read while it
    // still runs; its partials and LSEs only after the wait.
    bool act = false;
    float gam = 1.0f;
    if (mine) {
        act = p.window != 0 || p.active[row * p.act_s0] != 0;
        if (act && p.gate)
            gam = gate_factor(p.gate[(row / p.groups) * p.g_s0 +
                                     static_cast<int64_t>((row % p.groups) * p.heads + h) * p.g_s1]);
    }
    pdl_wait();   // partials come from the split kernel
    SDA_STAMP(threadIdx.x == 0 && blockIdx.x < kTimelineUnits, kTimelineCombine + blockIdx.x * 2ull + 1);
    if (!mine)
        return;
    uint16_t *out = p.output + static_cast<int64_t>(row) * p.o_s0 + static_cast<int64_t>(h) * p.o_s1 + d;
    if (!act) {
        if (p.clear_inactive)
            out[0] = out[1] = out[2] = out[3] = 0;
        return;
    }
    const int S = p.splits;
    const float *l = p.lse + static_cast<int64_t>(row) * S * p.heads + h;
    const float4 *part = reinterpret_cast<const float4 *>(
        p.partial + (static_cast<int64_t>(row) * S * p.heads + h) * kDim + d);
    const int64_t step = static_cast<int64_t>(p.heads) * (kDim / 4);   // float4s between splits
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    float wsum = 0.0f;
    // splits in groups of 4: a group's LSEs and partials load together
    float M = -INFINITY;
    for (int s = 0; s < S; ++s)
        M = S <= 4 ? M : fmaxf(M, l[s * p.heads]);
    for (int s0 = 0; s0 < S; s0 += 4) {
        float lv[4];
        float4 pv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            lv[j] = s0 + j < S ? l[(s0 + j) * p.heads] : -INFINITY;
            pv[j] = s0 + j < S ? part[(s0 + j) * step] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
        if (S <= 4)
            M = fmaxf(fmaxf(lv[0], lv[1]), fmaxf(lv[2], lv[3]));
        if (M == -INFINITY)
            break;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (lv[j] == -INFINITY)
                continue;
            const float w = expf(lv[j] - M);
            wsum += w;
            acc.x += w * pv[j].x;
            acc.y += w * pv[j].y;
            acc.z += w * pv[j].z;
            acc.w += w * pv[j].w;
        }
    }
    const float f = wsum > 0.0f ? gam / wsum : 0.0f;
    out[0] = __bfloat16_as_ushort(__float2bfloat16_rn(acc.x * f));
    out[1] = __bfloat16_as_ushort(__float2bfloat16_rn(acc.y * f));
    out[2] = __bfloat16_as_ushort(__float2bfloat16_rn(acc.z * f));
    out[3] = __bfloat16_as_ushort(__float2bfloat16_rn(acc.w * f));
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
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

std::atomic<unsigned long long> g_wait_ns{1000000000ull};

bool dims_ok(const sda_tensor *t, int ndim)
{
    if (!t || t->ndim != ndim)
        return false;
    for (int i = 0; i < ndim; ++i)
        if (t->shape[i] < 0)
            return false;
    return true;
}

// The dynamic shared memory limit each kernel instantiation has been raised to,
// per device.
template <bool FP8, bool WINDOW, bool FULL, bool PAIR>
cudaError_t ensure_smem(size_t bytes)
{
    static std::mutex mu;
    static size_t raised[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    std::lock_guard<std::mutex> lock(mu);
    size_t &cur = raised[dev & 63];
    if (bytes <= cur)
        return cudaSuccess;
    e = cudaFuncSetAttribute(sda_split_kernel<FP8, WINDOW, FULL, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(bytes));
    if (e == cudaSuccess)
        cur = bytes;
    return e;
}

template <bool FP8, bool WINDOW, bool FULL, bool PAIR = false>
sda_status launch(const CUtensorMap &tmap, const Params &prm, int num_regions, cudaStream_t stream)
{
    const size_t smem = Layout<FP8, PAIR>::bytes(num_regions);
    if (smem > 227 * 1024)
        return SDA_ERR_UNSUPPORTED;
    if (ensure_smem<FP8, WINDOW, FULL, PAIR>(smem) != cudaSuccess)
        return SDA_ERR_CUDA;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(PAIR ? prm.rows / 2 : prm.rows) * static_cast<unsigned>(prm.splits));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, sda_split_kernel<FP8, WINDOW, FULL, PAIR>, tmap, prm) != cudaSuccess)
        return SDA_ERR_CUDA;
    if (prm.splits > 1) {
        cudaLaunchConfig_t c2 = {};
        c2.gridDim = dim3(static_cast<unsigned>(prm.rows));
        c2.blockDim = dim3(static_cast<unsigned>(prm.heads * (kDim / 4)));
        c2.dynamicSmemBytes = 0;
        c2.stream = stream;
        c2.attrs = attr;
        c2.numAttrs = 1;
        if (cudaLaunchKernelEx(&c2, sda_combine_kernel, prm) != cudaSuccess)
            return SDA_ERR_CUDA;
    }
    return SDA_OK;
}

}  // namespace

// Read by the other translation units' kernels (hidden from the library's exports).
__attribute__((visibility("hidden"))) uint64_t sda_wait_limit_ns()
{
    return g_wait_ns.load();
}

extern "C" {

int sparse_decode_splits(int rows)
{
    int splits = 1;
    while (splits < 32 && static_cast<long long>(rows) * splits * 2 <= 256)
        splits *= 2;
    return rows < 0 ? 1 : splits;
}

size_t sparse_decode_workspace_bytes(int rows, int heads, int splits)
{
    if (rows < 0 || heads < 1 || heads > kMaxHeads || splits < 1 || splits > kMaxSplits)
        return 0;
    size_t bytes = kHeaderBytes;
    if (splits > 1) {
        const size_t n = static_cast<size_t>(rows) * splits * heads;
        bytes += n * kDim * sizeof(float);
        bytes += (n * sizeof(float) + 255) & ~static_cast<size_t>(255);
    }
    return bytes;
}

void sparse_decode_set_wait_limit_ns(uint64_t ns)
{
    g_wait_ns.store(ns);
}

const char *sparse_decode_status_string(int status)
{
    switch (status) {
    case SDA_OK: return "ok";
    case SDA_ERR_INVALID: return "invalid argument";
    case SDA_ERR_UNSUPPORTED: return "unsupported argument combination";
    case SDA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case SDA_ERR_CUDA: return "CUDA call failed";
    case SDA_ERR_TIMEOUT: return "a bounded device wait timed out";
    case SDA_ERR_BOUNDS: return "an index read from the inputs was out of range";
    default: return "unknown status";
    }
}

sda_status sparse_decode_timeline_buffer(void *buffer, size_t bytes)
{
#ifdef SDA_TIMELINE
    if (buffer && bytes < kTimelineBytes)
        return SDA_ERR_INVALID;
    unsigned long long *ptr = static_cast<unsigned long long *>(buffer);
    return cudaMemcpyToSymbol(g_sda_timeline, &ptr, sizeof ptr) == cudaSuccess ? SDA_OK : SDA_ERR_CUDA;
#else
    (void)buffer;
    (void)bytes;
    return SDA_ERR_UNSUPPORTED;
#endif
}

sda_status sparse_decode_read_errors(const void *workspace, uint32_t *flags, int clear, void *stream)
{
    if (!workspace || !flags)
        return SDA_ERR_INVALID;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t host = 0;
    if (cudaMemcpyAsync(&host, workspace, sizeof host, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return SDA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess)
        return SDA_ERR_CUDA;
    *flags = host;
    if (clear) {
        if (cudaMemsetAsync(const_cast<void *>(workspace), 0, sizeof host, s) != cudaSuccess)
            return SDA_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess)
            return SDA_ERR_CUDA;
    }
    return SDA_OK;
}

}  // extern "C"

namespace {

// One call of either entry point after argument unpacking.  Sparse mode uses
// regions / positions / active; window mode (window > 0) uses seq_lens.
struct Call {
    const sda_tensor *query, *cache, *regions, *block_table, *positions, *active, *seq_lens, *output, *gate;
    float scale;
    int query_len, splits, clear_inactive, region_tokens, window;
    const float *k_scale, *v_scale;
    void *workspace;
    size_t workspace_bytes;
    void *stream;
};

// With check_only, returns after the argument contract (everything but the
// workspace) without touching the GPU.
sda_status run_call(const Call &c, bool check_only = false)
{
    const bool windowed = c.window > 0;
    const sda_tensor *query = c.query, *cache = c.cache, *block_table = c.block_table, *output = c.output;
    // ---- Shape / dtype / stride contract (the page's asserts and the
    // eligibility test of the direct sparse decode path).
    if (!dims_ok(query, 3) || !dims_ok(cache, 4) || !dims_ok(block_table, 2) || !dims_ok(output, 3))
        return SDA_ERR_INVALID;
    const int64_t rows = query->shape[0], heads = query->shape[1];
    if (query->dtype != SDA_DTYPE_BF16 || output->dtype != SDA_DTYPE_BF16)
        return SDA_ERR_INVALID;
    if (query->shape[2] != kDim || cache->shape[3] != kRow)
        return SDA_ERR_INVALID;
    if (heads < 1 || heads > kMaxHeads)
        return SDA_ERR_UNSUPPORTED;
    if (output->shape[0] != rows || output->shape[1] != heads || output->shape[2] != kDim)
        return SDA_ERR_INVALID;
    if (query->stride[2] != 1 || output->stride[2] != 1 || cache->stride[3] != 1)
        return SDA_ERR_INVALID;
    if (block_table->dtype != SDA_DTYPE_INT32 || block_table->stride[1] != 1)
        return SDA_ERR_INVALID;
    if (windowed) {
        if (!dims_ok(c.seq_lens, 1) || c.seq_lens->dtype != SDA_DTYPE_INT32 || c.window > (1 << 30))
            return SDA_ERR_INVALID;
    } else {
        const sda_tensor *regions = c.regions, *positions = c.positions, *active = c.active;
        if (!dims_ok(regions, 2) || !dims_ok(positions, 1) || !dims_ok(active, 1))
            return SDA_ERR_INVALID;
        if (regions->dtype != SDA_DTYPE_INT32 || regions->shape[0] != rows || regions->stride[1] != 1)
            return SDA_ERR_INVALID;
        if (positions->dtype != SDA_DTYPE_INT32 || positions->shape[0] != rows)
            return SDA_ERR_INVALID;
        if ((active->dtype != SDA_DTYPE_BOOL && active->dtype != SDA_DTYPE_UINT8) || active->shape[0] != rows)
            return SDA_ERR_INVALID;
        if (regions->shape[1] > (1 << 14))
            return SDA_ERR_UNSUPPORTED;
    }
    const bool fp8 = cache->dtype == SDA_DTYPE_FP8_E4M3 || cache->dtype == SDA_DTYPE_UINT8;
    if (!fp8 && cache->dtype != SDA_DTYPE_BF16)
        return SDA_ERR_INVALID;
    if (fp8 && (!c.k_scale || !c.v_scale))
        return SDA_ERR_INVALID;
    if (c.query_len < 1 || c.splits < 1 || c.splits > kMaxSplits || !std::isfinite(c.scale))
        return SDA_ERR_INVALID;
    const int64_t pages = cache->shape[0], groups = cache->shape[1], block = cache->shape[2];
    if (groups < 1 || block < 1 || pages < 1 || pages > INT32_MAX)
        return SDA_ERR_INVALID;
    if (rows % groups != 0)
        return SDA_ERR_INVALID;
    const int64_t per_req = groups * c.query_len;
    const int64_t requests = rows > 0 ? (rows + per_req - 1) / per_req : 0;
    if (requests > block_table->shape[0] || (windowed && requests > c.seq_lens->shape[0]))
        return SDA_ERR_INVALID;
    const sda_tensor *gate = c.gate;
    const bool gated = gate && gate->data;
    if (gated) {
        if (!dims_ok(gate, 2) || gate->dtype != SDA_DTYPE_BF16 || gate->shape[0] != rows / groups ||
            gate->shape[1] != groups * heads)
            return SDA_ERR_INVALID;
    }
    const int64_t stage_tokens = fp8 ? Traits<true>::kSlots : Traits<false>::kSlots;
    int64_t rt, piece;
    if (windowed) {                        // the window is walked in pieces of P tokens
        piece = std::min<int64_t>(block, stage_tokens);
        rt = piece;
        if (piece % 8 != 0 || block % piece != 0)
            return SDA_ERR_UNSUPPORTED;
    } else {
        rt = c.region_tokens == 0 ? block : c.region_tokens;
        if (rt < 1 || rt > (1 << 24))
            return SDA_ERR_INVALID;
        piece = std::min<int64_t>(std::min<int64_t>(rt, block), stage_tokens);
        if (piece % 8 != 0 || rt % piece != 0 || block % piece != 0)
            return SDA_ERR_UNSUPPORTED;
    }
    if (block_table->shape[1] > INT32_MAX || rows > INT32_MAX / kMaxSplits)
        return SDA_ERR_UNSUPPORTED;
    // TMA: 16-byte aligned base and byte strides.
    const int elt = fp8 ? 1 : 2;
    const uintptr_t cbase = reinterpret_cast<uintptr_t>(cache->data);
    if (cbase % 16 != 0 || (cache->stride[0] * elt) % 16 != 0 || (cache->stride[1] * elt) % 16 != 0 ||
        (cache->stride[2] * elt) % 16 != 0 || cache->stride[0] <= 0 || cache->stride[1] <= 0 ||
        cache->stride[2] <= 0)
        return SDA_ERR_UNSUPPORTED;
    if (check_only)
        return SDA_OK;
    const size_t need = sparse_decode_workspace_bytes(static_cast<int>(rows), static_cast<int>(heads), c.splits);
    if (!c.workspace || reinterpret_cast<uintptr_t>(c.workspace) % 256 != 0 || c.workspace_bytes < need)
        return SDA_ERR_WORKSPACE;
    if (rows == 0)
        return SDA_OK;
    if (!query->data || !cache->data || !block_table->data || !output->data)
        return SDA_ERR_INVALID;
    if (windowed ? !c.seq_lens->data : (!c.regions->data || !c.positions->data || !c.active->data))
        return SDA_ERR_INVALID;

    // ---- Tensor map over the whole cache as (128-byte band chunk, token, band,
    // group, page): one box of 128 bytes x P tokens x all bands is a whole
    // piece, landing as [band][token][128 bytes] with 128-byte swizzle.
    EncodeTiledFn encode = encode_fn();
    if (!encode)
        return SDA_ERR_CUDA;
    CUtensorMap tmap;
    const int bands = kRow * elt / 128;
    const cuuint64_t gdim[5] = {static_cast<cuuint64_t>(128 / elt), static_cast<cuuint64_t>(block),
                                static_cast<cuuint64_t>(bands), static_cast<cuuint64_t>(groups),
                                static_cast<cuuint64_t>(pages)};
    const cuuint64_t gstride[4] = {static_cast<cuuint64_t>(cache->stride[2] * elt), 128u,
                                   static_cast<cuuint64_t>(cache->stride[1] * elt),
                                   static_cast<cuuint64_t>(cache->stride[0] * elt)};
    const cuuint32_t box[5] = {static_cast<cuuint32_t>(128 / elt), static_cast<cuuint32_t>(piece),
                               static_cast<cuuint32_t>(bands), 1, 1};
    const cuuint32_t estride[5] = {1, 1, 1, 1, 1};
    if (encode(&tmap, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5,
               const_cast<void *>(cache->data), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return SDA_ERR_UNSUPPORTED;

    Params prm;
    std::memset(&prm, 0, sizeof prm);
    prm.query = static_cast<const uint16_t *>(query->data);
    prm.q_s0 = query->stride[0];
    prm.q_s1 = query->stride[1];
    if (!windowed) {
        prm.regions = static_cast<const int32_t *>(c.regions->data);
        prm.reg_s0 = c.regions->stride[0];
        prm.num_regions = static_cast<int>(c.regions->shape[1]);
        prm.positions = static_cast<const int32_t *>(c.positions->data);
        prm.pos_s0 = c.positions->stride[0];
        prm.active = static_cast<const uint8_t *>(c.active->data);
        prm.act_s0 = c.active->stride[0];
    } else {
        prm.seq_lens = static_cast<const int32_t *>(c.seq_lens->data);
        prm.window = c.window;
    }
    prm.block_table = static_cast<const int32_t *>(block_table->data);
    prm.bt_s0 = block_table->stride[0];
    prm.output = static_cast<uint16_t *>(const_cast<void *>(output->data));
    prm.o_s0 = output->stride[0];
    prm.o_s1 = output->stride[1];
    prm.gate = gated ? static_cast<const uint16_t *>(gate->data) : nullptr;
    prm.g_s0 = gated ? gate->stride[0] : 0;
    prm.g_s1 = gated ? gate->stride[1] : 0;
    prm.k_scale = c.k_scale;
    prm.v_scale = c.v_scale;
    uint8_t *ws = static_cast<uint8_t *>(c.workspace);
    prm.flags = reinterpret_cast<unsigned int *>(ws);
    if (c.splits > 1) {
        const size_t n = static_cast<size_t>(rows) * c.splits * heads;
        prm.partial = reinterpret_cast<float *>(ws + kHeaderBytes);
        prm.lse = reinterpret_cast<float *>(ws + kHeaderBytes + n * kDim * sizeof(float));
    }
    prm.pages = pages;
    prm.wait_ns = g_wait_ns.load();
    prm.scale = c.scale;
    prm.table_cols = static_cast<int>(block_table->shape[1]);
    prm.rows = static_cast<int>(rows);
    prm.heads = static_cast<int>(heads);
    prm.groups = static_cast<int>(groups);
    prm.block = static_cast<int>(block);
    prm.region_tokens = static_cast<int>(rt);
    prm.piece = static_cast<int>(piece);
    prm.query_len = c.query_len;
    prm.splits = c.splits;
    prm.clear_inactive = c.clear_inactive ? 1 : 0;

    cudaStream_t s = static_cast<cudaStream_t>(c.stream);
    const int nr = windowed ? 0 : prm.num_regions;
    const bool full = piece == stage_tokens;
    // Window rows come in token pairs of one request (query_len even): one CTA
    // streams (its split's share of) the pair's union window once.
    const bool pair = windowed && c.query_len % 2 == 0;
    if (fp8) {
        if (pair)
            return full ? launch<true, true, true, true>(tmap, prm, nr, s)
                        : launch<true, true, false, true>(tmap, prm, nr, s);
        if (windowed)
            return full ? launch<true, true, true>(tmap, prm, nr, s) : launch<true, true, false>(tmap, prm, nr, s);
        return full ? launch<true, false, true>(tmap, prm, nr, s) : launch<true, false, false>(tmap, prm, nr, s);
    }
    if (pair)
        return full ? launch<false, true, true, true>(tmap, prm, nr, s)
                    : launch<false, true, false, true>(tmap, prm, nr, s);
    if (windowed)
        return full ? launch<false, true, true>(tmap, prm, nr, s) : launch<false, true, false>(tmap, prm, nr, s);
    return full ? launch<false, false, true>(tmap, prm, nr, s) : launch<false, false, false>(tmap, prm, nr, s);
}

}  // namespace

extern "C" {

sda_status sparse_decode_attention(const sda_tensor *query, const sda_tensor *cache,
                                   const sda_tensor *regions, const sda_tensor *block_table,
                                   const sda_tensor *positions, const sda_tensor *active,
                                   const sda_tensor *output, float scale, int query_len,
                                   int splits, const float *k_scale, const float *v_scale,
                                   const sda_tensor *gate, int clear_inactive, int region_tokens,
                                   void *workspace, size_t workspace_bytes, void *stream)
{
    if (!regions || !positions || !active)
        return SDA_ERR_INVALID;
    const Call c{query, cache, regions, block_table, positions, active, nullptr, output, gate,
                 scale, query_len, splits, clear_inactive, region_tokens, 0,
                 k_scale, v_scale, workspace, workspace_bytes, stream};
    return run_call(c);
}

int sparse_decode_swa_splits(int rows, int window)
{
    int splits = sparse_decode_splits(rows);
    while (splits > 1 && window / splits < 256)
        splits /= 2;
    return splits;
}

sda_status sparse_decode_swa_attention(const sda_tensor *query, const sda_tensor *cache,
                                       const sda_tensor *block_table, const sda_tensor *seq_lens,
                                       const sda_tensor *output, float scale, int window, int query_len,
                                       int splits, const float *k_scale, const float *v_scale,
                                       const sda_tensor *gate, void *workspace, size_t workspace_bytes,
                                       void *stream)
{
    if (!seq_lens || window < 1)
        return SDA_ERR_INVALID;
    const Call c{query, cache, nullptr, block_table, nullptr, nullptr, seq_lens, output, gate,
                 scale, query_len, splits, 1, 0, window,
                 k_scale, v_scale, workspace, workspace_bytes, stream};
    return run_call(c);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free entry point.
//
// For callers that hold device pointers to their tensors but have no way to
// obtain more device memory: plugin or FFI hosts that receive buffers from
// another runtime without an allocator handle, and code that must not call
// cudaMalloc while other work is in flight (an allocation can synchronise the
// device).  The split-KV scratch (flag header, fp32 partials and LSEs) lives
// in the fixed file-scope array below instead of a caller-supplied buffer.
// Every GPU that loads this library holds the array until the process exits.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;   // 8 MiB per device
static __device__ __align__(256) unsigned char g_sda_static_scratch[kStaticScratchBytes];

std::mutex g_static_scratch_mu;
void *g_static_scratch_ptr[256] = {};   // device address of the array, per device

// The array's device address on the current device.  The first use on a device
// looks it up (cudaGetSymbolAddress, with that device current) and zeroes the
// flag header on `stream`; later uses only read the cached address.
sda_status static_scratch(cudaStream_t stream, void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return SDA_ERR_CUDA;
    if (dev < 0 || dev >= 256)
        return SDA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_static_scratch_mu);
    if (!g_static_scratch_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_sda_static_scratch) != cudaSuccess || !ptr)
            return SDA_ERR_CUDA;
        if (cudaMemsetAsync(ptr, 0, kHeaderBytes, stream) != cudaSuccess)
            return SDA_ERR_CUDA;
        g_static_scratch_ptr[dev] = ptr;
    }
    *out = g_static_scratch_ptr[dev];
    return SDA_OK;
}

}  // namespace

extern "C" sda_status sparse_decode_attention_no_alloc(
    const sda_tensor *query, const sda_tensor *cache, const sda_tensor *regions,
    const sda_tensor *block_table, const sda_tensor *positions, const sda_tensor *active,
    const sda_tensor *output, float scale, int query_len, int splits, const float *k_scale,
    const float *v_scale, const sda_tensor *gate, int clear_inactive, int region_tokens, void *stream)
{
    if (!regions || !positions || !active)
        return SDA_ERR_INVALID;
    Call c{query, cache, regions, block_table, positions, active, nullptr, output, gate,
           scale, query_len, splits, clear_inactive, region_tokens, 0,
           k_scale, v_scale, nullptr, 0, stream};
    // The argument contract first, with the statuses of the regular entry
    // point; then the one status of this variant: scratch beyond the array.
    if (const sda_status st = run_call(c, true))
        return st;
    const size_t need = sparse_decode_workspace_bytes(static_cast<int>(query->shape[0]),
                                                      static_cast<int>(query->shape[1]), splits);
    if (need == 0 || need > kStaticScratchBytes)
        return SDA_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (const sda_status st = static_scratch(s, &c.workspace))
        return st;
    // The kernels only OR into the flag header, so flags collect over calls
    // until sparse_decode_no_alloc_read_errors clears them; partials and LSEs
    // are written before they are read and need no clearing.
    c.workspace_bytes = kStaticScratchBytes;
    return run_call(c);
}

extern "C" sda_status sparse_decode_no_alloc_read_errors(uint32_t *flags, int clear, void *stream)
{
    if (!flags)
        return SDA_ERR_INVALID;
    void *scratch = nullptr;
    if (const sda_status st = static_scratch(static_cast<cudaStream_t>(stream), &scratch))
        return st;
    return sparse_decode_read_errors(scratch, flags, clear, stream);
}
