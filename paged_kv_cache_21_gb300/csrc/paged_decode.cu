// paged_decode_attention: one decode step of attention over a block-paged KV
// cache, for sm_103a.
//
// What is computed: for each sequence s and query head h (KV head h / G),
//     out[s][h] = softmax_j(scale * q[s][h] . K_j) V_j,   j < context_lens[s]
// ("KV Cache" (heepie.pages.dev), section "Self-Attention"; the length mask of
// "Transformer attention mask and KV cache inference", section "Padding mask
// and batch length"), with K_j / V_j reached through the sequence's block
// table ("KV Cache, Flash Attention and inference optimization", section
// "PagedAttention").  The softmax is the running (max, sum) form that the
// same lesson's section "Numerical trick" shows to be exact.
//
// How (GB300 design):
//  * The step is HBM-bound: every (block, KV head) tile is read exactly once.
//    The flat list of all (sequence, KV head, block) units is cut into equal
//    contiguous ranges, one per warp of a persistent grid sized from the SM
//    count and measured occupancy, so every warp streams the same number of
//    bytes whatever the mix of context lengths (split-KV).
//  * Each warp owns a private ring of stages.  Its lane 0 fetches a block's
//    K and V tiles with TMA (cp.async.bulk.tensor, 128-byte swizzle) onto an
//    mbarrier; the ring keeps several tiles in flight per warp.  Block-table
//    entries for the next 32 blocks are fetched one window ahead.
//  * One MMA per 16-token block and k-step covers the whole GQA group: the
//    query rows of the G heads (padded to the 16-row MMA tile) times K^T,
//    then P (the running-softmax weights, kept in registers; for bf16 split
//    into a bf16 high and low part so they carry ~16 bits) times V.  The C
//    fragment of the score MMA is exactly the B fragment of the PV MMA, so
//    scores never leave registers.
//  * Warps whose range covers a whole (sequence, KV head) write the output
//    directly; the others store an unnormalised partial output with its
//    (max, sum) -- plain stores, no atomics or fences, so the split kernel
//    ends as soon as its last tile is consumed -- and a small merge kernel
//    combines them by the log-sum-exp rule in warp order (deterministic).
//    Both kernels use programmatic dependent launch: each is launched while
//    the previous kernel on the stream drains and waits on the device
//    (griddepcontrol.wait) before touching memory, which hides the launch
//    latency between them.
//  * Optionally (paged_decode_step) the append of the step's new token is
//    fused in: the warp that owns a pair's last block writes the new K/V to
//    the cache and patches its own copy of that tile in shared memory before
//    using it.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>

#include "device_common.cuh"
#include "internal.h"
#include "paged_kv.h"

namespace pkv {

__device__ DevErr g_decode_err;

constexpr int kWarps = 4;                        // warps per CTA (independent pipelines)
// Shared memory given to each warp's ring of stages, and the CTAs per SM the
// register allocation must allow, per KV element type.
constexpr int kWarpStageBytesBf16 = 24576;
constexpr int kWarpStageBytesFp8 = 24576;
constexpr int kMinCtasBf16 = 1;
constexpr int kMinCtasFp8 = 1;
constexpr int kMinBlocksPerWarp = 16;            // do not split below 256 tokens per warp
constexpr long long kWaitLimit = 1LL << 31;      // ~1 s of SM clocks

template <int D, bool FP8>
struct Geom {
    static constexpr int ES = FP8 ? 1 : 2;                    // element bytes
    static constexpr int ROWB = D * ES;                       // bytes per token row
    static constexpr int BOXW = ROWB >= 128 ? 128 : ROWB;     // bytes per TMA box row
    static constexpr int NBOX = ROWB / BOXW;                  // boxes per tile
    static constexpr int BOXB = kBlock * BOXW;                // bytes per box
    static constexpr int TILE = kBlock * ROWB;                // one (block, head) tile
    static constexpr int STAGE = 2 * TILE;                    // K + V
    static constexpr int STAGES_RAW = (FP8 ? kWarpStageBytesFp8 : kWarpStageBytesBf16) / STAGE;
    static constexpr int MIN_CTAS = FP8 ? kMinCtasFp8 : kMinCtasBf16;
    static constexpr int STAGES = STAGES_RAW < 2 ? 2 : (STAGES_RAW > 8 ? 8 : STAGES_RAW);
    static constexpr int SWZ = BOXW == 128 ? 7 : 3;           // 128B or 64B swizzle
    static constexpr int KSTEPS = D / 16;
    static constexpr int MTILES = D / 16;
    static constexpr int CHUNKS_PER_BOXROW = BOXW / 16;
    // shared memory: [stages of every warp][mbarriers][stage metadata (int4)],
    // the stage area aligned to 1024 bytes for the swizzled bulk copies
    static constexpr int BAR_OFF = kWarps * STAGES * STAGE;
    static constexpr int META_OFF = (BAR_OFF + kWarps * STAGES * 8 + 15) / 16 * 16;
    static constexpr int SMEM = META_OFF + kWarps * STAGES * 16 + 1024;
    static_assert(TILE % 1024 == 0 && BOXB % 512 == 0, "swizzled tiles need aligned stages");
    static_assert(BAR_OFF % 8 == 0 && META_OFF % 16 == 0, "barrier / metadata alignment");
    static_assert(SMEM <= 232448, "shared memory per CTA");
};

// Byte offset inside a tile of 16-byte chunk `c` of token row `r`, after the
// TMA swizzle (chunk bits XOR row bits of the 1024/512-byte pattern).
template <class G>
__device__ __forceinline__ uint32_t tile_off(int r, int c)
{
    const int box = c / G::CHUNKS_PER_BOXROW;
    const int cc = c % G::CHUNKS_PER_BOXROW;
    const uint32_t a = (uint32_t)(r * G::BOXW + cc * 16);
    return (uint32_t)(box * G::BOXB) + (a ^ (((a >> 7) & G::SWZ) << 4));
}

struct DecodeParams {
    const uint16_t* q;       // bf16 [B][Hq][D]
    void* out;               // [B][Hq][D] bf16 or f32
    const int32_t* bt;       // [B][max_blocks]
    const int32_t* ctx;      // [B]
    float* part_o;           // [slots][G][D]
    float2* part_ml;         // [slots][G]  (max in log2 units, sum)
    int2* pair_meta;         // [B*Hkv]  (first warp, number of partials)
    const uint16_t* k_new;   // bf16 [B][Hkv][D], or null: no append
    const uint16_t* v_new;
    uint8_t* k_cache;        // caches, written only by the fused append
    uint8_t* v_cache;
    int B, Hq, Hkv, G, max_blocks, num_blocks;
    int warps_total;
    float sl2;               // scale * log2(e) (* k_scale)
    float v_scale;
    float k_qscale, v_qscale;    // quantisation scales of the fused append (E4M3)
    int out_f32;
};

__device__ __forceinline__ int warp_incl_scan(int v, int lane)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(kFull, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

__device__ __forceinline__ int warp_sum(int v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// Context length of sequence s clamped to its block-table row; returns the
// number of blocks.
__device__ __forceinline__ int seq_blocks(const int32_t* ctx, int s, int max_blocks, int& Lc)
{
    int L = __ldg(ctx + s);
    const int cap = max_blocks * kBlock;
    if (L < 0 || L > cap) {
        raise_flag(&g_decode_err, KV_DEVERR_CONTEXT_TOO_LONG, L);
        L = L < 0 ? 0 : cap;
    }
    Lc = L;
    return (L + kBlock - 1) / kBlock;
}

// One lane's entry of the block-id window.
struct Win {
    int id, s, h, blk, L;
};

// Fill the window for flat positions pos0 + lane (relative to the warp's
// range start), walking forward from cursor (s, h, blk) where blk may equal
// the pair's block count (then the walk moves on to the next pair).
__device__ __forceinline__ void fill_window(Win& e, const DecodeParams& p, int s, int h, int blk,
                                            int nb, int L, int pos0, int cnt, int lane)
{
    e.id = -1; e.s = 0; e.h = 0; e.blk = 0; e.L = 0;
    if (pos0 + lane >= cnt) return;
    int r = lane;
    while (r >= nb - blk) {
        r -= nb - blk;
        blk = 0;
        if (++h == p.Hkv) {
            h = 0;
            do {
                if (++s >= p.B) return;      // inconsistent input: leave the entry invalid
                nb = seq_blocks(p.ctx, s, p.max_blocks, L);
            } while (nb == 0);
        }
    }
    blk += r;
    e.id = __ldg(p.bt + (size_t)s * p.max_blocks + blk);
    e.s = s; e.h = h; e.blk = blk; e.L = L;
}

// Four E4M3 codes (bytes 0..3 of w) -> two f16x2: lo = (byte0, byte1), hi =
// (byte2, byte3), each element exact (E4M3 is a subset of f16).  The word
// is split into its 16-bit halves so each conversion reads a register half.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi)
{
    asm("{\n\t.reg .b16 l, h;\n\t"
        "mov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

// Row d of the O^T accumulator held in fragment element (m-tile i, half).
template <int D, bool FP8>
__device__ __forceinline__ int out_dim(int i, int g, int half)
{
    if (FP8) return (D / 8) * g + 2 * i + half;
    return 16 * i + 8 * half + g;
}

// ------------------------------------------------------------ per-block math

// Online-softmax update over NBK consecutive blocks of one pair, from each
// block's scores of this lane's head (lane / 4) at tokens (2t, 2t+1, 2t+8,
// 2t+9); only the last block may be partial (nvalid_last tokens).  Returns
// the probabilities of those tokens and rescales the accumulator.
template <int D, int NBK>
__device__ __forceinline__ void softmax_update(const float (&sc)[NBK][2][4], int nvalid_last,
                                               float sl2, float& m, float& l,
                                               float (&o)[D / 16][4], float (&pr)[NBK][4],
                                               int lane)
{
    const int t = lane & 3;
    float x[NBK][4];
#pragma unroll
    for (int j = 0; j < NBK; ++j) {
        x[j][0] = sc[j][0][0] * sl2;
        x[j][1] = sc[j][0][1] * sl2;
        x[j][2] = sc[j][1][0] * sl2;
        x[j][3] = sc[j][1][1] * sl2;
    }
    if (nvalid_last < kBlock) {
        const int t0 = 2 * t;
        if (t0 >= nvalid_last) x[NBK - 1][0] = -INFINITY;
        if (t0 + 1 >= nvalid_last) x[NBK - 1][1] = -INFINITY;
        if (t0 + 8 >= nvalid_last) x[NBK - 1][2] = -INFINITY;
        if (t0 + 9 >= nvalid_last) x[NBK - 1][3] = -INFINITY;
    }
    float mx = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[0][2], x[0][3]));
#pragma unroll
    for (int j = 1; j < NBK; ++j)
        mx = fmaxf(mx, fmaxf(fmaxf(x[j][0], x[j][1]), fmaxf(x[j][2], x[j][3])));
    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
    const float m_new = fmaxf(m, mx);
    const float alpha = exp2f(m - m_new);
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < NBK; ++j) {
        pr[j][0] = exp2f(x[j][0] - m_new);
        pr[j][1] = exp2f(x[j][1] - m_new);
        pr[j][2] = exp2f(x[j][2] - m_new);
        pr[j][3] = exp2f(x[j][3] - m_new);
        sum += (pr[j][0] + pr[j][1]) + (pr[j][2] + pr[j][3]);
    }
    l = l * alpha + sum;
    m = m_new;
    // accumulator columns are heads 2t and 2t+1: fetch their factors
    const float aa = __shfl_sync(kFull, alpha, 8 * t);
    const float ab = __shfl_sync(kFull, alpha, 8 * t + 4);
    if (__any_sync(kFull, aa != 1.f || ab != 1.f)) {
#pragma unroll
        for (int i = 0; i < D / 16; ++i) {
            o[i][0] *= aa;
            o[i][1] *= ab;
            o[i][2] *= aa;
            o[i][3] *= ab;
        }
    }
}

// Scores q.K of the 16 tokens of one bf16 tile: sc[0] tokens 0-7, sc[1]
// tokens 8-15 (C fragments: row = head, column = token).
template <int D>
__device__ __forceinline__ void scores_bf16(uint32_t kbase, const uint32_t (&qa0)[D / 16],
                                            const uint32_t (&qa2)[D / 16], float (&sc)[2][4],
                                            int lane)
{
    using G = Geom<D, false>;
    const int mi = lane >> 3, ri = lane & 7;
    const int tok = ri + 8 * (mi >> 1);
    const int csel = mi & 1;
#pragma unroll
    for (int k = 0; k < 4; ++k) sc[0][k] = sc[1][k] = 0.f;
#pragma unroll
    for (int s = 0; s < G::KSTEPS; ++s) {
        uint32_t r[4];
        ldsm_x4(r, kbase + tile_off<G>(tok, 2 * s + csel));
        mma_bf16(sc[0], qa0[s], 0u, qa2[s], 0u, r[0], r[1]);
        mma_bf16(sc[1], qa0[s], 0u, qa2[s], 0u, r[2], r[3]);
    }
}

// O^T += V^T P^T for one bf16 tile; P is split into bf16 hi + lo parts.
template <int D>
__device__ __forceinline__ void pv_bf16(uint32_t vbase, int nvalid, const float (&pr)[4],
                                        float (&o)[D / 16][4], int lane)
{
    using G = Geom<D, false>;
    const int t = lane & 3;
    const int mi = lane >> 3, ri = lane & 7;
    const int tok = ri + 8 * (mi >> 1);
    const int csel = mi & 1;
    const uint32_t h0 = pack_bf16x2(pr[0], pr[1]);
    const uint32_t h1 = pack_bf16x2(pr[2], pr[3]);
    const uint32_t e0 = pack_bf16x2(pr[0] - bf16_lo(h0), pr[1] - bf16_hi(h0));
    const uint32_t e1 = pack_bf16x2(pr[2] - bf16_lo(h1), pr[3] - bf16_hi(h1));
    uint32_t m01 = 0xffffffffu, m23 = 0xffffffffu;
    if (nvalid < kBlock) {      // zero V rows past the context (they may hold anything)
        const int t0 = 2 * t;
        m01 = (t0 < nvalid ? 0x0000ffffu : 0u) | (t0 + 1 < nvalid ? 0xffff0000u : 0u);
        m23 = (t0 + 8 < nvalid ? 0x0000ffffu : 0u) | (t0 + 9 < nvalid ? 0xffff0000u : 0u);
    }
#pragma unroll
    for (int i = 0; i < G::MTILES; ++i) {
        uint32_t r[4];
        ldsm_x4_trans(r, vbase + tile_off<G>(tok, 2 * i + csel));
        r[0] &= m01; r[1] &= m01; r[2] &= m23; r[3] &= m23;
        mma_bf16(o[i], r[0], r[1], r[2], r[3], h0, h1);
        mma_bf16(o[i], r[0], r[1], r[2], r[3], e0, e1);
    }
}

// Scores of one E4M3 tile: bytes via ldmatrix, widened to f16 in registers.
template <int D>
__device__ __forceinline__ void scores_fp8(uint32_t kbase, const uint32_t (&qa0)[D / 16],
                                           const uint32_t (&qa2)[D / 16], float (&sc)[2][4],
                                           int lane)
{
    using G = Geom<D, true>;
    const int mi = lane >> 3, ri = lane & 7;
    const int tok = ri + 8 * (mi & 1);
    const int csel = mi >> 1;
#pragma unroll
    for (int k = 0; k < 4; ++k) sc[0][k] = sc[1][k] = 0.f;
#pragma unroll
    for (int c = 0; c < G::KSTEPS; c += 2) {
        uint32_t r[4];
        ldsm_x4(r, kbase + tile_off<G>(tok, c + csel));
        uint32_t b[4][2];
#pragma unroll
        for (int j = 0; j < 4; ++j) e4m3x4_to_f16x2x2(r[j], b[j][0], b[j][1]);
        mma_f16(sc[0], qa0[c], 0u, qa2[c], 0u, b[0][0], b[0][1]);
        mma_f16(sc[1], qa0[c], 0u, qa2[c], 0u, b[1][0], b[1][1]);
        mma_f16(sc[0], qa0[c + 1], 0u, qa2[c + 1], 0u, b[2][0], b[2][1]);
        mma_f16(sc[1], qa0[c + 1], 0u, qa2[c + 1], 0u, b[3][0], b[3][1]);
    }
}

// O^T += V^T P^T for one E4M3 tile; P in f16.
template <int D>
__device__ __forceinline__ void pv_fp8(uint32_t vbase, int nvalid, const float (&pr)[4],
                                       float (&o)[D / 16][4], int lane)
{
    using G = Geom<D, true>;
    const int g = lane >> 2, t = lane & 3;
    const uint32_t pf0 = pack_f16x2(pr[0], pr[1]);
    const uint32_t pf1 = pack_f16x2(pr[2], pr[3]);
    // V rows of tokens 2t, 2t+1, 2t+8, 2t+9, bytes [BYTES*g, BYTES*g + BYTES)
    constexpr int BYTES = D / 8;
    constexpr int WORDS = BYTES / 4;
    const int boff = BYTES * g;
    uint32_t x[4][WORDS];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int tk = 2 * t + (k & 1) + 8 * (k >> 1);
        const uint32_t a = vbase + tile_off<G>(tk, boff >> 4) + (boff & 15);
        if (WORDS == 4) {
            uint32_t r[4];
            lds128(r, a);
#pragma unroll
            for (int w = 0; w < WORDS; ++w) x[k][w] = r[w];
        } else {
            uint32_t r[2];
            lds64(r, a);
#pragma unroll
            for (int w = 0; w < WORDS; ++w) x[k][w] = r[w];
        }
        if (tk >= nvalid) {
#pragma unroll
            for (int w = 0; w < WORDS; ++w) x[k][w] = 0u;
        }
    }
#pragma unroll
    for (int w = 0; w < WORDS; ++w) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const uint32_t sel = e ? 0x7362u : 0x5140u;
            uint32_t a[4];
            e4m3x4_to_f16x2x2(__byte_perm(x[0][w], x[1][w], sel), a[0], a[1]);
            e4m3x4_to_f16x2x2(__byte_perm(x[2][w], x[3][w], sel), a[2], a[3]);
            mma_f16(o[2 * w + e], a[0], a[1], a[2], a[3], pf0, pf1);
        }
    }
}

// NBK consecutive tiles of one pair (K at kb[j], V right after it): scores
// of every tile first, one softmax update over all of them, then P.V.
template <int D, bool FP8, int NBK>
__device__ __forceinline__ void attend_tiles(const uint32_t (&kb)[NBK], int nvalid_last,
                                             const uint32_t (&qa0)[D / 16],
                                             const uint32_t (&qa2)[D / 16], float sl2, float& m,
                                             float& l, float (&o)[D / 16][4], int lane)
{
    using G = Geom<D, FP8>;
    float sc[NBK][2][4];
#pragma unroll
    for (int j = 0; j < NBK; ++j) {
        if (FP8) scores_fp8<D>(kb[j], qa0, qa2, sc[j], lane);
        else scores_bf16<D>(kb[j], qa0, qa2, sc[j], lane);
    }
    float pr[NBK][4];
    softmax_update<D, NBK>(sc, nvalid_last, sl2, m, l, o, pr, lane);
#pragma unroll
    for (int j = 0; j < NBK; ++j) {
        const int nv = j == NBK - 1 ? nvalid_last : kBlock;
        if (FP8) pv_fp8<D>(kb[j] + G::TILE, nv, pr[j], o, lane);
        else pv_bf16<D>(kb[j] + G::TILE, nv, pr[j], o, lane);
    }
}

// Query fragments of head (h*G + g) of sequence s (rows g >= G are zero).
template <int D, bool FP8>
__device__ __forceinline__ void load_q(const DecodeParams& p, int s, int h, int lane,
                                       uint32_t (&qa0)[D / 16], uint32_t (&qa2)[D / 16])
{
    const int g = lane >> 2, t = lane & 3;
    const bool live = g < p.G;
    const uint16_t* qh = p.q + ((size_t)s * p.Hq + (size_t)h * p.G + (live ? g : 0)) * D;
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
        if (!FP8) {
            const uint32_t* q32 = reinterpret_cast<const uint32_t*>(qh);
            qa0[k] = live ? __ldg(q32 + 8 * k + t) : 0u;
            qa2[k] = live ? __ldg(q32 + 8 * k + 4 + t) : 0u;
        } else {
            uint2 v = make_uint2(0u, 0u);
            if (live) v = __ldg(reinterpret_cast<const uint2*>(qh + 16 * k + 4 * t));
            qa0[k] = pack_f16x2(bf16_lo(v.x), bf16_hi(v.x));
            qa2[k] = pack_f16x2(bf16_lo(v.y), bf16_hi(v.y));
        }
    }
}

__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <class P>
__device__ __forceinline__ void store4(const P& p, size_t idx, float a, float b, float c, float d)
{
    if (p.out_f32) {
        *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + idx) = make_float4(a, b, c, d);
    } else {
        uint2 v;
        v.x = pack_bf16x2(a, b);
        v.y = pack_bf16x2(c, d);
        *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.out) + idx) = v;
    }
}

// End of a segment (a run of blocks of one pair inside this warp's range):
// write the final output if the warp saw the whole pair, otherwise store a
// partial for the merge kernel.  The warp holding the pair's block 0 also
// records which warps hold the rest.  Only plain stores: a pair switch in
// mid-range does not stall the warp's pipeline.
template <int D, bool FP8>
__device__ __forceinline__ void finalize(const DecodeParams& p, int w, int q, int s, int h,
                                         int first_blk, int last_blk, int L, int flat_first,
                                         float m, float l, const float (&o)[D / 16][4], int lane)
{
    const int g = lane >> 2, t = lane & 3;
    float lt = l + __shfl_xor_sync(kFull, l, 1);
    lt += __shfl_xor_sync(kFull, lt, 2);
    const float la = __shfl_sync(kFull, lt, 8 * t), lb = __shfl_sync(kFull, lt, 8 * t + 4);
    const float ma = __shfl_sync(kFull, m, 8 * t), mb = __shfl_sync(kFull, m, 8 * t + 4);
    const int nb = (L + kBlock - 1) / kBlock;
    const int pair = s * p.Hkv + h;
    const int ha = 2 * t, hb = 2 * t + 1;
    if (first_blk == 0 && last_blk == nb - 1) {
        const float ia = la > 0.f ? p.v_scale / la : 0.f;
        const float ib = lb > 0.f ? p.v_scale / lb : 0.f;
        const size_t row = (size_t)s * p.Hq + (size_t)h * p.G;
#pragma unroll
        for (int i = 0; i < D / 16; ++i) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int d = out_dim<D, FP8>(i, g, half);
                if (ha < p.G) {
                    const float v = o[i][2 * half] * ia;
                    const size_t idx = (row + ha) * D + d;
                    if (p.out_f32) reinterpret_cast<float*>(p.out)[idx] = v;
                    else reinterpret_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16_rn(v);
                }
                if (hb < p.G) {
                    const float v = o[i][2 * half + 1] * ib;
                    const size_t idx = (row + hb) * D + d;
                    if (p.out_f32) reinterpret_cast<float*>(p.out)[idx] = v;
                    else reinterpret_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16_rn(v);
                }
            }
        }
    } else {
        const size_t slot = (size_t)pair + w;
        float* po = p.part_o + slot * p.G * D;
#pragma unroll
        for (int i = 0; i < D / 16; ++i) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int d = out_dim<D, FP8>(i, g, half);
                if (ha < p.G) po[ha * D + d] = o[i][2 * half] * p.v_scale;
                if (hb < p.G) po[hb * D + d] = o[i][2 * half + 1] * p.v_scale;
            }
        }
        if (g == 0) {
            if (ha < p.G) p.part_ml[slot * p.G + ha] = make_float2(ma, la);
            if (hb < p.G) p.part_ml[slot * p.G + hb] = make_float2(mb, lb);
        }
    }
    if (first_blk == 0 && lane == 0) {
        // block 0 of the pair is here: record the warps whose ranges meet its
        // blocks [flat_first, flat_first + nb)
        const int w_last = (flat_first + nb - 1) / q;
        p.pair_meta[pair] = make_int2(w, w_last - w + 1);
    }
}

// The fused append of the step's new token of pair (s, h): position L-1,
// i.e. row (L-1) % 16 of the pair's last block `id`.  Writes the cache in
// global memory and the same bytes into this warp's copy of the tile in
// shared memory (which the bulk copy may have filled before the write).
template <int D, bool FP8>
__device__ __forceinline__ void append_patch(const DecodeParams& p, int s, int h, int id, int L,
                                             uint32_t kst, uint32_t vst, int lane)
{
    using G = Geom<D, FP8>;
    constexpr int CH = D / 8;              // groups of 8 elements per row
    if (lane < 2 * CH) {
        const bool isv = lane >= CH;
        const int c = isv ? lane - CH : lane;
        const int r = (L - 1) & (kBlock - 1);
        const size_t src = ((size_t)s * p.Hkv + h) * D + 8 * c;
        const size_t dst = (((size_t)id * p.Hkv + h) * kBlock + r) * D + 8 * c;
        const uint4 x = __ldg(reinterpret_cast<const uint4*>((isv ? p.v_new : p.k_new) + src));
        uint8_t* cache = isv ? p.v_cache : p.k_cache;
        const uint32_t sb = isv ? vst : kst;
        if (!FP8) {
            *reinterpret_cast<uint4*>(cache + dst * 2) = x;
            sts128(sb + tile_off<G>(r, c), x);
        } else {
            const uint2 y = quantize8_e4m3(x, isv ? p.v_qscale : p.k_qscale);
            *reinterpret_cast<uint2*>(cache + dst) = y;
            sts64(sb + tile_off<G>(r, c >> 1) + 8 * (c & 1), y);
        }
    }
    __syncwarp();
}

template <int D, bool FP8>
__global__ void __launch_bounds__(kWarps * 32, Geom<D, FP8>::MIN_CTAS)
paged_decode_split_kernel(const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const DecodeParams p)
{
    using G = Geom<D, FP8>;
    constexpr int ST = G::STAGES;
    extern __shared__ uint8_t smem_raw[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int w = blockIdx.x * kWarps + warp;

    const uint32_t sraw = smem_u32(smem_raw);
    const uint32_t sbase = (sraw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (sbase - sraw);
    const uint32_t stage0 = sbase + (uint32_t)(warp * ST * G::STAGE);
    const uint32_t bar0 = sbase + (uint32_t)(G::BAR_OFF + warp * ST * 8);
    int4* meta = reinterpret_cast<int4*>(gbase + G::META_OFF) + warp * ST;

    if (threadIdx.x == 0) {
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    // let the next kernel on the stream launch now, then wait until the
    // previous one has finished and its writes are visible
    pdl_launch_dependents();
    pdl_wait();

    // ---- 1. total work and this warp's range --------------------------------
    constexpr int U = 8;           // first 256 sequences stay in registers
    int nbv[U], incl[U];
    int carry = 0;
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int s = u * 32 + lane;
        int Lc;
        nbv[u] = s < p.B ? seq_blocks(p.ctx, s, p.max_blocks, Lc) : 0;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
        incl[u] = warp_incl_scan(nbv[u] * p.Hkv, lane) + carry;
        carry = __shfl_sync(kFull, incl[u], 31);
    }
    int total = carry;
    // sequences past the first 256: 256 at a time, all loads issued together
    for (int base = U * 32; base < p.B; base += U * 32) {
        int v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int s = base + u * 32 + lane;
            int Lc;
            v[u] = s < p.B ? seq_blocks(p.ctx, s, p.max_blocks, Lc) : 0;
        }
        int sum = 0;
#pragma unroll
        for (int u = 0; u < U; ++u) sum += v[u];
        total += warp_sum(sum) * p.Hkv;
    }
    if (total == 0) return;
    int q = (total + p.warps_total - 1) / p.warps_total;
    if (q < kMinBlocksPerWarp) q = kMinBlocksPerWarp;
    const int weff = (total + q - 1) / q;
    if (w >= weff) return;
    const int b0 = w * q;
    const int cnt = min(q, total - b0);

    // ---- 2. the (sequence, head, block) where the range starts --------------
    int s0 = -1, excl = 0;
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const unsigned mball = __ballot_sync(kFull, incl[u] > b0);
        if (s0 < 0 && mball) {
            const int src = __ffs(mball) - 1;
            s0 = u * 32 + src;
            excl = __shfl_sync(kFull, incl[u] - nbv[u] * p.Hkv, src);
        }
    }
    if (s0 < 0) {
        int c2 = carry;
        for (int base = U * 32; base < p.B && s0 < 0; base += U * 32) {
            int v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int s = base + u * 32 + lane;
                int Lc;
                v[u] = s < p.B ? seq_blocks(p.ctx, s, p.max_blocks, Lc) * p.Hkv : 0;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int inc = warp_incl_scan(v[u], lane) + c2;
                const unsigned mball = __ballot_sync(kFull, inc > b0);
                if (s0 < 0 && mball) {
                    const int src = __ffs(mball) - 1;
                    s0 = base + u * 32 + src;
                    excl = __shfl_sync(kFull, inc - v[u], src);
                }
                c2 = __shfl_sync(kFull, inc, 31);
            }
        }
    }
    if (s0 < 0) return;      // unreachable with consistent input
    int L0;
    const int nb0 = seq_blocks(p.ctx, s0, p.max_blocks, L0);
    const int off0 = b0 - excl;
    const int h0 = off0 / nb0;
    const int blk0 = off0 - h0 * nb0;

    // ---- 3. pipeline set-up ---------------------------------------------------
    if (lane == 0) {
#pragma unroll
        for (int st = 0; st < ST; ++st) mbar_init(bar0 + st * 8, 1);
        fence_mbar_init();
    }
    __syncwarp();

    Win cur, nxt;
    int wb = 0;
    fill_window(cur, p, s0, h0, blk0, nb0, L0, 0, cnt, lane);
    nxt = cur;
    auto refill_next = [&](int pos0) {
        const int cs = __shfl_sync(kFull, cur.s, 31), ch = __shfl_sync(kFull, cur.h, 31);
        const int cb = __shfl_sync(kFull, cur.blk, 31) + 1;
        const int cL = __shfl_sync(kFull, cur.L, 31);
        fill_window(nxt, p, cs, ch, cb, (cL + kBlock - 1) / kBlock, cL, pos0, cnt, lane);
    };
    if (cnt > 32) refill_next(32);

    auto issue = [&](int j, int st) {
        if (j >= wb + 32) {
            cur = nxt;
            wb += 32;
            if (wb + 32 < cnt) refill_next(wb + 32);
        }
        const int src = j - wb;
        const int id = __shfl_sync(kFull, cur.id, src);
        const int s = __shfl_sync(kFull, cur.s, src);
        const int h = __shfl_sync(kFull, cur.h, src);
        const int blk = __shfl_sync(kFull, cur.blk, src);
        const int L = __shfl_sync(kFull, cur.L, src);
        if (lane == 0) {
            const bool valid = id >= 0 && id < p.num_blocks;
            const int pair = s * p.Hkv + h;
            meta[st] = make_int4(valid ? pair : -1 - pair, blk, L, id);
            const uint32_t bar = bar0 + st * 8;
            const uint32_t dst = stage0 + (uint32_t)(st * G::STAGE);
            if (valid) {
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(bar, (uint32_t)G::STAGE);
                const int z = id * p.Hkv + h;
                // KV tiles are read once per step: keep them from evicting
                // the block tables, queries and partials from L2
                const uint64_t pol = l2_evict_first_policy();
#pragma unroll
                for (int b = 0; b < G::NBOX; ++b)
                    tma_load_3d_hint(dst + b * G::BOXB, &tm_k, b * (G::BOXW / G::ES), 0, z, bar,
                                     pol);
#pragma unroll
                for (int b = 0; b < G::NBOX; ++b)
                    tma_load_3d_hint(dst + G::TILE + b * G::BOXB, &tm_v, b * (G::BOXW / G::ES), 0,
                                     z, bar, pol);
            } else {
                raise_flag(&g_decode_err, KV_DEVERR_BLOCK_OUT_OF_RANGE, id);
                mbar_arrive(bar);
            }
        }
    };

    const int npro = min(ST, cnt);
    for (int j = 0; j < npro; ++j) issue(j, j);

    // ---- 4. main loop ------------------------------------------------------------
    // Two consecutive tiles of the same pair are consumed together where the
    // range allows: one softmax update and one loop turn per 32 tokens.
    uint32_t qa0[D / 16], qa2[D / 16];
    float o[D / 16][4];
    float m = -INFINITY, l = 0.f;
    int seg_s = -1, seg_h = -1, seg_first = 0, seg_last = 0, seg_L = 0, seg_i0 = 0;
    int seg_pair = -1;
    int st = 0;
    uint32_t phase = 0;
    // Wait for unit i in stage `sst`; on time-out flag the error and let the
    // copies of units [i, issued_end) land before the warp gives up.
    auto wait_unit = [&](int i, int sst, uint32_t ph, int issued_end) -> bool {
        bool ok = mbar_wait_bounded(bar0 + sst * 8, ph, kWaitLimit);
        ok = __all_sync(kFull, ok);
        if (!ok) {
            if (lane == 0) {
                raise_flag(&g_decode_err, KV_DEVERR_PIPELINE_TIMEOUT, i);
                for (int j = i; j < issued_end; ++j) {
                    mbar_wait_bounded(bar0 + sst * 8, ph, kWaitLimit);
                    if (++sst == ST) { sst = 0; ph ^= 1u; }
                }
            }
            __syncwarp();
        }
        return ok;
    };
    for (int i = 0; i < cnt;) {
        const int issued_end = min(cnt, i + ST);
        if (!wait_unit(i, st, phase, issued_end)) return;
        const int4 mt = meta[st];
        const bool valid = mt.x >= 0;
        const int pair = valid ? mt.x : -1 - mt.x;
        const int blk = mt.y, L = mt.z;
        if (pair != seg_pair) {
            seg_pair = pair;
            const int s = pair / p.Hkv, h = pair - s * p.Hkv;
            if (seg_s >= 0)
                finalize<D, FP8>(p, w, q, seg_s, seg_h, seg_first, seg_last, seg_L, b0 + seg_i0,
                                 m, l, o, lane);
            seg_s = s; seg_h = h; seg_first = blk; seg_L = L; seg_i0 = i;
            load_q<D, FP8>(p, s, h, lane, qa0, qa2);
            m = -INFINITY;
            l = 0.f;
#pragma unroll
            for (int a = 0; a < D / 16; ++a) o[a][0] = o[a][1] = o[a][2] = o[a][3] = 0.f;
        }
        const int st2 = st + 1 == ST ? 0 : st + 1;
        const uint32_t phase2 = st + 1 == ST ? phase ^ 1u : phase;
        bool two = false;
        if (valid && i + 1 < cnt) {
            __syncwarp();            // unit i+1's metadata was written by lane 0
            two = meta[st2].x == mt.x;
        }
        const uint32_t kb = stage0 + (uint32_t)(st * G::STAGE);
        if (two) {
            if (!wait_unit(i + 1, st2, phase2, issued_end)) return;
            const int id2 = meta[st2].w;
            const uint32_t kb2 = stage0 + (uint32_t)(st2 * G::STAGE);
            const int rest = L - (blk + 1) * kBlock;
            const int nvalid = min(kBlock, rest);
            if (p.k_new != nullptr && nvalid == rest)     // the pair's last block
                append_patch<D, FP8>(p, seg_s, seg_h, id2, L, kb2, kb2 + G::TILE, lane);
            const uint32_t kbs[2] = {kb, kb2};
            attend_tiles<D, FP8, 2>(kbs, nvalid, qa0, qa2, p.sl2, m, l, o, lane);
            seg_last = blk + 1;
            __syncwarp();
            if (i + ST < cnt) issue(i + ST, st);
            if (i + 1 + ST < cnt) issue(i + 1 + ST, st2);
            st = st2 + 1 == ST ? 0 : st2 + 1;
            phase = st2 + 1 == ST ? phase2 ^ 1u : phase2;
            i += 2;
        } else {
            seg_last = blk;
            if (valid) {
                const int nvalid = min(kBlock, L - blk * kBlock);
                if (p.k_new != nullptr && nvalid == L - blk * kBlock)     // the pair's last block
                    append_patch<D, FP8>(p, seg_s, seg_h, mt.w, L, kb, kb + G::TILE, lane);
                const uint32_t kbs[1] = {kb};
                attend_tiles<D, FP8, 1>(kbs, nvalid, qa0, qa2, p.sl2, m, l, o, lane);
            }
            __syncwarp();
            if (i + ST < cnt) issue(i + ST, st);
            st = st2;
            phase = phase2;
            i += 1;
        }
    }
    if (seg_s >= 0)
        finalize<D, FP8>(p, w, q, seg_s, seg_h, seg_first, seg_last, seg_L, b0 + seg_i0, m, l, o,
                         lane);
}

// -------------------------------------------------------------------- merge

struct MergeParams {
    void* out;
    const int32_t* ctx;
    const float* part_o;
    const float2* part_ml;
    const int2* pair_meta;
    int B, Hq, Hkv, G, max_blocks;
    int nslots;              // partial slots in the workspace
    int out_f32;
};

// One CTA per (sequence, KV head): merge the partials the split kernel left
// for it (pairs seen whole by one warp were written there already), or write
// zeros for an empty context.  Thread t owns output float4 column t of the
// pair's G x D block; the (max, sum) terms of up to 64 partials at a time go
// through shared memory, and a thread's partial loads are independent of one
// another, so the merge costs a few L2 round trips.
constexpr int kMergeThreads = 256;   // >= 8 heads x 128 / 4 columns
constexpr int kMergeChunk = 64;

template <int D>
__global__ void __launch_bounds__(kMergeThreads, 1) paged_decode_merge_kernel(const MergeParams p)
{
    __shared__ float2 sml[kMergeChunk * 8];
    pdl_launch_dependents();
    pdl_wait();
    const int pair = blockIdx.x;
    const int s = pair / p.Hkv, h = pair - s * p.Hkv;
    const int t = threadIdx.x;
    const int cols = p.G * (D / 4);
    const size_t row = (size_t)s * p.Hq + (size_t)h * p.G;
    int L;
    seq_blocks(p.ctx, s, p.max_blocks, L);
    if (L <= 0) {
        if (t < cols) store4(p, row * D + 4 * t, 0.f, 0.f, 0.f, 0.f);
        return;
    }
    const int2 mt = p.pair_meta[pair];
    const int n = mt.y;
    if (n <= 1) return;
    // the table is rewritten by every split launch; refuse anything that
    // would leave the workspace (only an aborted split launch leaves it stale)
    if (mt.x < 0 || (long long)pair + mt.x + n > (long long)p.nslots) return;
    const size_t slot0 = (size_t)pair + mt.x;
    const int g = t / (D / 4), d4 = t % (D / 4);
    const bool live = t < cols;
    float M = -INFINITY, den = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k0 = 0; k0 < n; k0 += kMergeChunk) {
        const int nk = min(kMergeChunk, n - k0);
        __syncthreads();
        for (int i = t; i < nk * p.G; i += kMergeThreads) {
            const int kk = i / p.G, gg = i - kk * p.G;
            float2 v = __ldcg(&p.part_ml[(slot0 + k0 + kk) * p.G + gg]);
            if (!(v.y > 0.f)) v = make_float2(-INFINITY, 0.f);     // empty partial
            sml[kk * 8 + gg] = v;
        }
        __syncthreads();
        if (!live) continue;
        float cm = -INFINITY;
        for (int k = 0; k < nk; ++k) cm = fmaxf(cm, sml[k * 8 + g].x);
        const float Mn = fmaxf(M, cm);
        const float r = Mn == -INFINITY ? 0.f : exp2f(M - Mn);
        den *= r;
        acc.x *= r; acc.y *= r; acc.z *= r; acc.w *= r;
        M = Mn;
        const float4* po = reinterpret_cast<const float4*>(p.part_o + (slot0 + k0) * p.G * D) +
                           (size_t)g * (D / 4) + d4;
#pragma unroll 8
        for (int k = 0; k < nk; ++k) {
            const float4 o = __ldcg(po + (size_t)k * p.G * (D / 4));
            const float2 v = sml[k * 8 + g];
            const float f = v.y > 0.f ? exp2f(v.x - M) : 0.f;
            den += f * v.y;
            acc.x += f * o.x;
            acc.y += f * o.y;
            acc.z += f * o.z;
            acc.w += f * o.w;
        }
    }
    if (live) {
        const float inv = den > 0.f ? 1.f / den : 0.f;
        store4(p, (row + g) * D + 4 * d4, acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
}

// ------------------------------------------------------------------- host

namespace {

constexpr int kMaxDevices = 64;

struct VariantInfo {
    bool ready = false;
    int ctas_per_sm = 0;
};

struct DeviceInfo {
    bool ready = false;
    int sms = 0;
    VariantInfo v[2][2];    // [D==128][fp8]
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

template <int D, bool FP8>
const void* split_fn()
{
    return reinterpret_cast<const void*>(&paged_decode_split_kernel<D, FP8>);
}

template <int D, bool FP8>
int variant_setup(VariantInfo& vi)
{
    using G = Geom<D, FP8>;
    const void* fn = split_fn<D, FP8>();
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM) !=
        cudaSuccess)
        return KV_ERR_CUDA;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kWarps * 32, G::SMEM) !=
            cudaSuccess ||
        n <= 0)
        return KV_ERR_CUDA;
    vi.ctas_per_sm = n;
    vi.ready = true;
    return KV_OK;
}

// Device facts and per-variant occupancy, cached per device.
int device_info(int D, bool fp8, int& sms, int& ctas_per_sm)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KV_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo& di = g_dev[dev];
    if (!di.ready) {
        if (cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return KV_ERR_CUDA;
        di.ready = true;
    }
    VariantInfo& vi = di.v[D == 128][fp8];
    if (!vi.ready) {
        int rc;
        if (D == 128) rc = fp8 ? variant_setup<128, true>(vi) : variant_setup<128, false>(vi);
        else rc = fp8 ? variant_setup<64, true>(vi) : variant_setup<64, false>(vi);
        if (rc != KV_OK) return rc;
    }
    sms = di.sms;
    ctas_per_sm = vi.ctas_per_sm;
    return KV_OK;
}

int tensor_map_encoder(PFN_cuTensorMapEncodeTiled_v12000& fn)
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !ptr)
            return KV_ERR_CUDA;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    fn = g_encode;
    return KV_OK;
}

// Tensor map over a cache viewed as [num_blocks*Hkv][16][D]; one box is 16
// token rows x (128 or 64) bytes, swizzled to match tile_off().
int make_cache_map(CUtensorMap* map, const void* base, int D, bool fp8, int num_blocks, int Hkv)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    if (int rc = tensor_map_encoder(enc)) return rc;
    const int es = fp8 ? 1 : 2;
    const int rowb = D * es;
    const int boxw = rowb >= 128 ? 128 : rowb;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)kBlock, (cuuint64_t)num_blocks * Hkv};
    cuuint64_t strides[2] = {(cuuint64_t)rowb, (cuuint64_t)rowb * kBlock};
    cuuint32_t box[3] = {(cuuint32_t)(boxw / es), (cuuint32_t)kBlock, 1u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUresult r = enc(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                           3, const_cast<void*>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE,
                           boxw == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? KV_OK : KV_ERR_CUDA;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
    size_t part_o, part_ml, meta, total;
};

WsLayout ws_layout(int B, int Hq, int Hkv, int D, int warps_total)
{
    const int G = Hq / Hkv;
    const size_t slots = (size_t)B * Hkv + (size_t)warps_total;
    WsLayout L;
    L.part_o = 0;
    L.part_ml = align256(slots * G * D * sizeof(float));
    L.meta = L.part_ml + align256(slots * G * sizeof(float2));
    L.total = L.meta + align256((size_t)B * Hkv * sizeof(int2));
    return L;
}

int check_shape(int num_seqs, int Hq, int Hkv, int D, int kv_dtype)
{
    if (num_seqs < 0 || Hq <= 0 || Hkv <= 0) return KV_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return KV_ERR_INVALID_ARG;
    const int G = Hq / Hkv;
    if (G > 8) return KV_ERR_UNSUPPORTED;
    if (D != 64 && D != 128) return KV_ERR_UNSUPPORTED;
    if (kv_dtype != KV_DTYPE_BF16 && kv_dtype != KV_DTYPE_FP8_E4M3) return KV_ERR_UNSUPPORTED;
    return KV_OK;
}

// Launch with programmatic stream serialisation: the kernel may start while
// the previous kernel on the stream drains; it waits on the device
// (griddepcontrol.wait) before touching memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                       cudaStream_t st, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

struct AppendArgs {
    const void* k_new;
    const void* v_new;
    void* k_cache;
    void* v_cache;
};

// Validate, build the tensor maps and launch the decode kernel (one launch).
int decode_launch(void* out, int out_dtype, const void* q, const void* k_cache,
                  const void* v_cache, int kv_dtype, float k_scale, float v_scale, int num_blocks,
                  const int32_t* block_tables, int max_blocks_per_seq,
                  const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                  int head_dim, float scale, void* workspace, size_t workspace_bytes,
                  void* stream, const AppendArgs* app, void* ev_begin, void* ev_split,
                  void* ev_end)
{
    if (int rc = check_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, kv_dtype)) return rc;
    if (out_dtype != KV_DTYPE_BF16 && out_dtype != KV_DTYPE_F32) return KV_ERR_UNSUPPORTED;
    if (num_seqs == 0) return KV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !workspace)
        return KV_ERR_INVALID_ARG;
    if (num_blocks <= 0 || max_blocks_per_seq <= 0) return KV_ERR_INVALID_ARG;
    if ((((uintptr_t)q | (uintptr_t)k_cache | (uintptr_t)v_cache | (uintptr_t)workspace |
          (uintptr_t)out) & 15) != 0)
        return KV_ERR_INVALID_ARG;
    if (app && (!app->k_new || !app->v_new ||
                (((uintptr_t)app->k_new | (uintptr_t)app->v_new) & 15) != 0))
        return KV_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return KV_ERR_INVALID_ARG;
    const bool fp8 = kv_dtype == KV_DTYPE_FP8_E4M3;
    if (fp8 && !(k_scale > 0.f && v_scale > 0.f && std::isfinite(k_scale) && std::isfinite(v_scale)))
        return KV_ERR_INVALID_ARG;
    // flat work indices and tensor-map rows must fit in int32
    if ((long long)num_seqs * max_blocks_per_seq * num_kv_heads >= INT_MAX ||
        (long long)num_blocks * num_kv_heads >= INT_MAX ||
        (long long)max_blocks_per_seq * kBlock >= INT_MAX)
        return KV_ERR_UNSUPPORTED;

    int sms = 0, cps = 0;
    if (int rc = device_info(head_dim, fp8, sms, cps)) return rc;
    const int grid = sms * cps;
    const int warps_total = grid * kWarps;
    const WsLayout ws = ws_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, warps_total);
    if (workspace_bytes < ws.total) return KV_ERR_INVALID_ARG;

    CUtensorMap mk, mv;
    if (int rc = make_cache_map(&mk, k_cache, head_dim, fp8, num_blocks, num_kv_heads)) return rc;
    if (int rc = make_cache_map(&mv, v_cache, head_dim, fp8, num_blocks, num_kv_heads)) return rc;

    uint8_t* wsb = static_cast<uint8_t*>(workspace);
    DecodeParams dp;
    dp.q = static_cast<const uint16_t*>(q);
    dp.out = out;
    dp.bt = block_tables;
    dp.ctx = context_lens;
    dp.part_o = reinterpret_cast<float*>(wsb + ws.part_o);
    dp.part_ml = reinterpret_cast<float2*>(wsb + ws.part_ml);
    dp.pair_meta = reinterpret_cast<int2*>(wsb + ws.meta);
    dp.k_new = app ? static_cast<const uint16_t*>(app->k_new) : nullptr;
    dp.v_new = app ? static_cast<const uint16_t*>(app->v_new) : nullptr;
    dp.k_cache = app ? static_cast<uint8_t*>(app->k_cache) : nullptr;
    dp.v_cache = app ? static_cast<uint8_t*>(app->v_cache) : nullptr;
    dp.B = num_seqs;
    dp.Hq = num_q_heads;
    dp.Hkv = num_kv_heads;
    dp.G = num_q_heads / num_kv_heads;
    dp.max_blocks = max_blocks_per_seq;
    dp.num_blocks = num_blocks;
    dp.warps_total = warps_total;
    dp.sl2 = scale * 1.4426950408889634f * (fp8 ? k_scale : 1.f);
    dp.v_scale = fp8 ? v_scale : 1.f;
    dp.k_qscale = k_scale;
    dp.v_qscale = v_scale;
    dp.out_f32 = out_dtype == KV_DTYPE_F32;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (ev_begin && cudaEventRecord(static_cast<cudaEvent_t>(ev_begin), st) != cudaSuccess)
        return KV_ERR_CUDA;
    const int threads = kWarps * 32;
    cudaError_t err;
    if (head_dim == 128) {
        if (fp8)
            err = launch_pdl(paged_decode_split_kernel<128, true>, grid, threads,
                             Geom<128, true>::SMEM, st, mk, mv, dp);
        else
            err = launch_pdl(paged_decode_split_kernel<128, false>, grid, threads,
                             Geom<128, false>::SMEM, st, mk, mv, dp);
    } else {
        if (fp8)
            err = launch_pdl(paged_decode_split_kernel<64, true>, grid, threads,
                             Geom<64, true>::SMEM, st, mk, mv, dp);
        else
            err = launch_pdl(paged_decode_split_kernel<64, false>, grid, threads,
                             Geom<64, false>::SMEM, st, mk, mv, dp);
    }
    if (err != cudaSuccess) return KV_ERR_CUDA;
    if (ev_split && cudaEventRecord(static_cast<cudaEvent_t>(ev_split), st) != cudaSuccess)
        return KV_ERR_CUDA;

    MergeParams mp;
    mp.out = out;
    mp.ctx = context_lens;
    mp.part_o = dp.part_o;
    mp.part_ml = dp.part_ml;
    mp.pair_meta = dp.pair_meta;
    mp.B = num_seqs;
    mp.Hq = num_q_heads;
    mp.Hkv = num_kv_heads;
    mp.G = dp.G;
    mp.max_blocks = max_blocks_per_seq;
    mp.nslots = num_seqs * num_kv_heads + warps_total;
    mp.out_f32 = dp.out_f32;
    const unsigned mgrid = (unsigned)(num_seqs * num_kv_heads);
    err = head_dim == 128
              ? launch_pdl(paged_decode_merge_kernel<128>, mgrid, kMergeThreads, 0, st, mp)
              : launch_pdl(paged_decode_merge_kernel<64>, mgrid, kMergeThreads, 0, st, mp);
    if (err != cudaSuccess) return KV_ERR_CUDA;
    if (ev_end && cudaEventRecord(static_cast<cudaEvent_t>(ev_end), st) != cudaSuccess)
        return KV_ERR_CUDA;
    return KV_OK;
}

}  // namespace

int num_sms_current()
{
    int dev = 0, n = 1;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev >= 0 && dev < kMaxDevices) {
        std::lock_guard<std::mutex> lk(g_mu);
        if (g_dev[dev].ready) return g_dev[dev].sms;
    }
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
    return n;
}

int decode_read_error(unsigned* flags, long long* detail)
{
    DevErr e;
    if (cudaMemcpyFromSymbol(&e, g_decode_err, sizeof e) != cudaSuccess) return KV_ERR_CUDA;
    DevErr z = {0u, -1LL};
    if (cudaMemcpyToSymbol(g_decode_err, &z, sizeof z) != cudaSuccess) return KV_ERR_CUDA;
    *flags = e.flags;
    *detail = e.flags ? e.detail : -1;
    return KV_OK;
}

// ------------------------------------------------- fixed, library-owned scratch
// Scratch of the allocation-free entry point: a file-scope device array that
// every device loading the library holds until the process exits.  Host code
// must not use the symbol's name as an address: its device address is looked
// up once per device with cudaGetSymbolAddress (with that device current).
constexpr size_t kStaticWorkspaceBytes = 16u << 20;     // 16 MiB
__device__ __align__(256) uint8_t g_static_workspace[kStaticWorkspaceBytes];

namespace {

void* g_static_ws_ptr[kMaxDevices] = {};

// Device address of g_static_workspace on the current device (set up once).
int static_workspace(void** ptr)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KV_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_static_ws_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p) return KV_ERR_CUDA;
        g_static_ws_ptr[dev] = p;
    }
    *ptr = g_static_ws_ptr[dev];
    return KV_OK;
}

}  // namespace

}  // namespace pkv

using namespace pkv;

extern "C" int paged_decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                            int head_dim, int kv_dtype, size_t* bytes)
{
    if (!bytes) return KV_ERR_INVALID_ARG;
    *bytes = 0;
    if (int rc = check_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, kv_dtype)) return rc;
    int sms = 0, cps = 0;
    if (int rc = device_info(head_dim, kv_dtype == KV_DTYPE_FP8_E4M3, sms, cps)) return rc;
    *bytes = ws_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, sms * cps * kWarps).total;
    return KV_OK;
}

extern "C" int paged_decode_attention_timed(
    void* out, int out_dtype, const void* q, const void* k_cache, const void* v_cache,
    int kv_dtype, float k_scale, float v_scale, int num_blocks, const int32_t* block_tables,
    int max_blocks_per_seq, const int32_t* context_lens, int num_seqs, int num_q_heads,
    int num_kv_heads, int head_dim, float scale, void* workspace, size_t workspace_bytes,
    void* stream, void* ev_begin, void* ev_split_end, void* ev_end)
{
    return decode_launch(out, out_dtype, q, k_cache, v_cache, kv_dtype, k_scale, v_scale,
                         num_blocks, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                         num_q_heads, num_kv_heads, head_dim, scale, workspace, workspace_bytes,
                         stream, nullptr, ev_begin, ev_split_end, ev_end);
}

extern "C" int paged_decode_attention(void* out, int out_dtype, const void* q, const void* k_cache,
                                      const void* v_cache, int kv_dtype, float k_scale,
                                      float v_scale, int num_blocks, const int32_t* block_tables,
                                      int max_blocks_per_seq, const int32_t* context_lens,
                                      int num_seqs, int num_q_heads, int num_kv_heads,
                                      int head_dim, float scale, void* workspace,
                                      size_t workspace_bytes, void* stream)
{
    return decode_launch(out, out_dtype, q, k_cache, v_cache, kv_dtype, k_scale, v_scale,
                         num_blocks, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                         num_q_heads, num_kv_heads, head_dim, scale, workspace, workspace_bytes,
                         stream, nullptr, nullptr, nullptr, nullptr);
}

extern "C" int paged_decode_step(void* out, int out_dtype, const void* q, const void* k_new,
                                 const void* v_new, void* k_cache, void* v_cache, int kv_dtype,
                                 float k_scale, float v_scale, int num_blocks,
                                 const int32_t* block_tables, int max_blocks_per_seq,
                                 const int32_t* context_lens, int num_seqs, int num_q_heads,
                                 int num_kv_heads, int head_dim, float scale, void* workspace,
                                 size_t workspace_bytes, void* stream)
{
    const AppendArgs app = {k_new, v_new, k_cache, v_cache};
    return decode_launch(out, out_dtype, q, k_cache, v_cache, kv_dtype, k_scale, v_scale,
                         num_blocks, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                         num_q_heads, num_kv_heads, head_dim, scale, workspace, workspace_bytes,
                         stream, &app, nullptr, nullptr, nullptr);
}

extern "C" int kv_get_device_error(int* flags, int64_t* detail)
{
    unsigned f1 = 0, f2 = 0;
    long long d1 = -1, d2 = -1;
    if (int rc = append_read_error(&f1, &d1)) return rc;
    if (int rc = decode_read_error(&f2, &d2)) return rc;
    if (flags) *flags = (int)(f1 | f2);
    if (detail) *detail = f1 ? d1 : d2;
    return KV_OK;
}

extern "C" int paged_decode_attention_noalloc(void* out, int out_dtype, const void* q,
                                              const void* k_cache, const void* v_cache,
                                              int kv_dtype, float k_scale, float v_scale,
                                              int num_blocks, const int32_t* block_tables,
                                              int max_blocks_per_seq, const int32_t* context_lens,
                                              int num_seqs, int num_q_heads, int num_kv_heads,
                                              int head_dim, float scale, void* stream)
{
    if (int rc = check_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, kv_dtype)) return rc;
    if (num_seqs == 0) return KV_OK;
    size_t need = 0;
    if (int rc = paged_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                              kv_dtype, &need))
        return rc;
    if (need > kStaticWorkspaceBytes) return KV_ERR_TOO_LARGE;
    void* ws = nullptr;
    if (int rc = static_workspace(&ws)) return rc;
    return paged_decode_attention(out, out_dtype, q, k_cache, v_cache, kv_dtype, k_scale, v_scale,
                                  num_blocks, block_tables, max_blocks_per_seq, context_lens,
                                  num_seqs, num_q_heads, num_kv_heads, head_dim, scale, ws,
                                  kStaticWorkspaceBytes, stream);
}
