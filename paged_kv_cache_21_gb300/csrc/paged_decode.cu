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
//    scores never leave registers.  Two consecutive tiles of a pair are
//    consumed together where the range allows: one online-softmax update per
//    32 tokens.
//  * Warps whose range covers a whole (sequence, KV head) write the output
//    directly; the others store an unnormalised partial output with its
//    (max, sum) -- plain stores, no atomics or fences, so the split kernel
//    ends as soon as its last tile is consumed -- and a small merge kernel
//    combines them by the log-sum-exp rule in warp order (deterministic).
//    Both kernels use programmatic dependent launch: each is launched while
//    the previous kernel on the stream drains and waits on the device
//    (griddepcontrol.wait) before touching memory, which hides the launch
//    latency between them.  The merge kernel lets the next kernel start only
//    after its own wait, so with KV_DECODE_EARLY_INPUTS the next step's
//    split kernel can read its block tables and cache tiles before waiting.
//  * Optionally (paged_decode_step) the append of the step's new token is
//    fused in: the warp that owns a pair's last block writes the new K/V to
//    the cache and patches its own copy of that tile in shared memory before
//    using it.
//  * Query groups of 9-16 rows fill both 8-row halves of the MMA tile (the
//    two-row-tile kernel); larger groups (MQA on many-head models) run as
//    2^k sub-groups of <= 16 rows, one team of warps each, the teams cutting
//    the same units the same way so that a tile's repeated reads hit L2.
//  * Shared prefixes (paged_decode with a chunk table): sequences whose
//    block tables start with the same blocks ("KV cache complete guide",
//    sections "(3) Prefix Caching" and "(4) PagedAttention") are cut into
//    chunks whose query rows fill the whole 16-row MMA tile; each shared tile
//    is read once per chunk, and the merge kernel adds each member's rows of
//    the chunk's partials to its own.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>

#include "device_common.cuh"
#include "internal.h"
#include "paged_kv.h"
#include "wide.h"

namespace pkv {

__device__ DevErr g_decode_err;

// Warps per CTA (independent pipelines) per KV element type.
constexpr int kWarpsBf16 = 4;
constexpr int kWarpsFp8 = 4;
// Shared memory given to each warp's ring of stages, and the CTAs per SM the
// register allocation must allow, per KV element type.
constexpr int kWarpStageBytesBf16 = 24576;
constexpr int kWarpStageBytesFp8 = 24576;
constexpr int kMinCtasBf16 = 1;
constexpr int kMinCtasFp8 = 1;
// Minimum range of a warp.  Sequence phase: at most 16 blocks (256 tokens);
// with a narrow block table, ceil(max_blocks / 8) but at least 2, so that a
// small problem spreads over more warps while every pair still meets about
// kMergeDirect ranges (the merge's one-round-trip path).
constexpr int kMinBlocksPerWarp = 16;
constexpr int kMinBlocksPerWarpChunk = 4;        // the prefix chunk phase
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
    static constexpr int WARPS = FP8 ? kWarpsFp8 : kWarpsBf16;
    static constexpr int STAGES = STAGES_RAW < 2 ? 2 : (STAGES_RAW > 8 ? 8 : STAGES_RAW);
    static constexpr int SWZ = BOXW == 128 ? 7 : 3;           // 128B or 64B swizzle
    static constexpr int KSTEPS = D / 16;
    static constexpr int MTILES = D / 16;
    static constexpr int CHUNKS_PER_BOXROW = BOXW / 16;
    // shared memory: [stages of every warp][mbarriers][stage metadata (int4)],
    // the stage area aligned to 1024 bytes for the swizzled bulk copies
    static constexpr int BAR_OFF = WARPS * STAGES * STAGE;
    // one more barrier per warp that nothing arrives on (the time-out test hook)
    static constexpr int STALL_OFF = BAR_OFF + WARPS * STAGES * 8;
    static constexpr int META_OFF = (STALL_OFF + WARPS * 8 + 15) / 16 * 16;
    static constexpr int SMEM = META_OFF + WARPS * STAGES * 16 + 1024;
    static_assert(TILE % 1024 == 0 && BOXB % 512 == 0, "swizzled tiles need aligned stages");
    static_assert(BAR_OFF % 8 == 0 && STALL_OFF % 8 == 0 && META_OFF % 16 == 0,
                  "barrier / metadata alignment");
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
    float* part_o;           // [slots][prow][D]
    float2* part_ml;         // [slots][prow]  (max in log2 units, sum)
    int4* pair_meta;         // [streams*Hkv]  (first warp, number of partials,
                             //  the sequence's (chunk << 4 | member) or -1, 0)
    const uint16_t* k_new;   // bf16 [B][Hkv][D], or null: no append
    const uint16_t* v_new;
    uint8_t* k_cache;        // caches, written only by the fused append
    uint8_t* v_cache;
    // Hkv and G count virtual KV heads and their rows (groups above 16 rows
    // are cut into sub-groups, see hshift)
    int B, Hq, Hkv, G, max_blocks, num_blocks;
    int warps_total;
    int min_q1;              // minimum range of a warp in the sequence phase
    int hshift;              // a KV head serves 1 << hshift virtual heads of G rows
    int Hkv_p;               // physical KV heads (Hkv >> hshift)
    int team_slots;          // partial slots of one team: streams * Hkv_p + its warps
    float sl2;               // scale * log2(e) (* k_scale)
    float v_scale;
    float k_qscale, v_qscale;    // quantisation scales of the fused append (E4M3)
    int out_f32;
    const int32_t* chunk;        // prefix chunks [nc][KV_PREFIX_CHUNK_INTS]
    const int32_t* seq_chunk;    // [B]: (chunk << 4) | member index, or -1
    int nc;                      // number of prefix chunks
    int prow;                    // rows per partial slot
    int slot_base;               // first partial slot of the sequence phase
    int early;                   // read the host-made inputs and caches before the wait
    long long test_stall;        // > 0: test hook, see kv_test_pipeline_stall
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
// number of blocks.  The split kernel's helpers only read (no flag atomics,
// so the compiler can batch their loads); the merge kernel, which visits
// every sequence, reports bad entries (report = true).
__device__ __forceinline__ int seq_blocks(const int32_t* ctx, int s, int max_blocks, int& Lc,
                                          bool report = false)
{
    int L = __ldg(ctx + s);
    const int cap = max_blocks * kBlock;
    if (L < 0 || L > cap) {
        if (report) raise_flag(&g_decode_err, KV_DEVERR_CONTEXT_TOO_LONG, L);
        L = L < 0 ? 0 : cap;
    }
    Lc = L;
    return (L + kBlock - 1) / kBlock;
}

// ------------------------------------------------------------------ streams
//
// The work is a list of streams, each a run of blocks of one block-table row
// attended by a set of query rows, for every KV head.  Streams [0, nc) are
// the prefix chunks -- the P leading blocks that a chunk of sequences share,
// attended once for all the chunk's query rows (up to 16: NR == 2 kernels
// process these) -- and stream nc + s is sequence s from its first block
// past its chunk's P (from block 0 without shared prefixes; NR == 1 kernels).

struct Stream {
    int nblk;    // blocks (per KV head)
    int base;    // first block: index into the block-table row
    int row;     // sequence whose block-table row holds the blocks
    int L;       // tokens of that row that count (masking of the last block)
    int cj;      // sequence stream with a shared prefix: (chunk << 4) | member, else -1
};

// P of chunk c if its table row is usable (P in [0, max_blocks], 1..16
// members, at most 16 query rows, member 0 a valid sequence), else -1.
__device__ __forceinline__ int chunk_blocks(const int32_t* chunk, int c, int B, int G,
                                            int max_blocks, int& lead, int& members,
                                            bool report = false)
{
    const int32_t* row = chunk + (size_t)c * KV_PREFIX_CHUNK_INTS;
    const int P = __ldg(row);
    members = __ldg(row + 1);
    lead = __ldg(row + 2);
    if (P < 0 || P > max_blocks || members < 1 || members > KV_PREFIX_MAX_MEMBERS ||
        members * G > KV_PREFIX_MAX_ROWS || lead < 0 || lead >= B) {
        if (report) raise_flag(&g_decode_err, KV_DEVERR_BAD_PREFIX, c);
        return -1;
    }
    return P;
}

// Shared leading blocks of sequence s (context L): its chunk's P when the
// chunk is usable, s really is its member j, and the P blocks lie before the
// new token; otherwise 0 (s is then attended alone, from block 0).
__device__ __forceinline__ int prefix_of(const int32_t* chunk, const int32_t* seq_chunk, int nc,
                                         int B, int G, int max_blocks, int s, int L, int& c,
                                         int& j, bool report = false)
{
    const int sc = __ldg(seq_chunk + s);
    if (sc < 0) return 0;
    c = sc >> 4;
    j = sc & 15;
    int lead, members;
    const int P = c < nc ? chunk_blocks(chunk, c, B, G, max_blocks, lead, members) : -1;
    bool ok = P >= 0 && j < members &&
              __ldg(chunk + (size_t)c * KV_PREFIX_CHUNK_INTS + 2 + j) == s;
    if (ok && P > 0 && (L < 1 || P > (L - 1) / kBlock)) ok = false;
    if (!ok) {
        if (report) raise_flag(&g_decode_err, KV_DEVERR_BAD_PREFIX, s);
        return 0;
    }
    return P;
}

// Sub-groups of a KV head exist only in the two-row-tile kernel (a group
// above 16 rows leaves sub-groups of 9-16 rows), so the one-row-tile kernel
// folds them away at compile time.
template <int NR>
__device__ __forceinline__ int hshift_of(const DecodeParams& p)
{
    return NR == 2 ? p.hshift : 0;
}

template <int NR>
__device__ __forceinline__ int hkv_phys(const DecodeParams& p)
{
    return NR == 2 ? p.Hkv_p : p.Hkv;
}

template <int NR>
__device__ __forceinline__ Stream stream_at(const DecodeParams& p, int sigma)
{
    Stream r;
    if (NR == 2 && sigma < p.nc) {
        int lead, members;
        const int P = chunk_blocks(p.chunk, sigma, p.B, p.G, p.max_blocks, lead, members);
        r.nblk = P > 0 ? P : 0;
        r.base = 0;
        r.row = P > 0 ? lead : 0;
        r.L = r.nblk * kBlock;
        r.cj = -1;
        return r;
    }
    // (NR == 1 kernels run without prefix chunks: nc is 0 there)
    if constexpr (NR == 2) sigma -= p.nc;
    int L;
    const int nb = seq_blocks(p.ctx, sigma, p.max_blocks, L);
    r.row = sigma;
    r.L = L;
    r.base = 0;
    r.cj = -1;
    if (NR == 2 && p.nc > 0) {
        int c = 0, j = 0;
        r.base = prefix_of(p.chunk, p.seq_chunk, p.nc, p.B, p.G, p.max_blocks, sigma, L, c, j);
        if (r.base > 0) r.cj = (c << 4) | j;
    }
    r.nblk = nb - r.base;
    return r;
}

// One lane's entry of the block-id window.
struct Win {
    int id, s, h, blk, L;    // s: the stream; blk: index into its block-table row
    int base, row;           // the stream's first block and block-table row
};

// Fill the window for flat positions pos0 + lane (relative to the warp's
// range start), walking forward from stream sg, head h, block j of the
// stream (j may equal the stream's block count: the walk then moves on).
template <int NR>
__device__ __forceinline__ void fill_window(Win& e, const DecodeParams& p, int ns, int sg, int h,
                                            int j, Stream S, int pos0, int cnt, int lane)
{
    e.id = -1; e.s = 0; e.h = 0; e.blk = 0; e.L = 0; e.base = 0; e.row = 0;
    if (pos0 + lane >= cnt) return;
    int r = lane;
    while (r >= S.nblk - j) {
        r -= S.nblk - j;
        j = 0;
        if (++h == hkv_phys<NR>(p)) {
            h = 0;
            do {
                if (++sg >= ns) return;      // inconsistent input: leave the entry invalid
                S = stream_at<NR>(p, sg);
            } while (S.nblk <= 0);
        }
    }
    j += r;
    e.id = __ldg(p.bt + (size_t)S.row * p.max_blocks + S.base + j);
    e.s = sg; e.h = h; e.blk = S.base + j; e.L = S.L; e.base = S.base; e.row = S.row;
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
//
// A unit's query rows sit in the rows of the 16-row MMA A operand: rows 0-7
// always, rows 8-15 as well when NR == 2 (a prefix chunk with more than 8
// query rows).  Lane (g = lane/4, t = lane%4) holds, per 8-token half of a
// block, the scores of rows g (and g + 8) at tokens 2t and 2t+1.

// Online-softmax update over NBK consecutive blocks of one stream for the NR
// row tiles, from each block's scores (only the last block may be partial:
// nvalid_last tokens).  Returns the probabilities of the lane's tokens (2t,
// 2t+1, 2t+8, 2t+9) and rescales the accumulators.
template <int D, int NBK, int NR>
__device__ __forceinline__ void softmax_update(const float (&sc)[NBK][2][4], int nvalid_last,
                                               const float (&sl2)[NR], float (&m)[NR],
                                               float (&l)[NR], float (&o)[NR][D / 16][4],
                                               float (&pr)[NBK][NR][4], int lane)
{
    const int t = lane & 3;
    float x[NBK][NR][4];
#pragma unroll
    for (int j = 0; j < NBK; ++j) {
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            x[j][r][0] = sc[j][0][2 * r] * sl2[r];
            x[j][r][1] = sc[j][0][2 * r + 1] * sl2[r];
            x[j][r][2] = sc[j][1][2 * r] * sl2[r];
            x[j][r][3] = sc[j][1][2 * r + 1] * sl2[r];
        }
    }
    if (nvalid_last < kBlock) {
        const int t0 = 2 * t;
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            if (t0 >= nvalid_last) x[NBK - 1][r][0] = -INFINITY;
            if (t0 + 1 >= nvalid_last) x[NBK - 1][r][1] = -INFINITY;
            if (t0 + 8 >= nvalid_last) x[NBK - 1][r][2] = -INFINITY;
            if (t0 + 9 >= nvalid_last) x[NBK - 1][r][3] = -INFINITY;
        }
    }
    float alpha[NR];
    bool rescale = false;
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        float mx = fmaxf(fmaxf(x[0][r][0], x[0][r][1]), fmaxf(x[0][r][2], x[0][r][3]));
#pragma unroll
        for (int j = 1; j < NBK; ++j)
            mx = fmaxf(mx, fmaxf(fmaxf(x[j][r][0], x[j][r][1]), fmaxf(x[j][r][2], x[j][r][3])));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
        const float m_new = fmaxf(m[r], mx);
        alpha[r] = exp2f(m[r] - m_new);
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < NBK; ++j) {
            pr[j][r][0] = exp2f(x[j][r][0] - m_new);
            pr[j][r][1] = exp2f(x[j][r][1] - m_new);
            pr[j][r][2] = exp2f(x[j][r][2] - m_new);
            pr[j][r][3] = exp2f(x[j][r][3] - m_new);
            sum += (pr[j][r][0] + pr[j][r][1]) + (pr[j][r][2] + pr[j][r][3]);
        }
        l[r] = l[r] * alpha[r] + sum;
        m[r] = m_new;
        rescale = rescale || alpha[r] != 1.f;
    }
    // accumulator columns are rows 2t and 2t+1 (+ 8r): fetch their factors
    if (__any_sync(kFull, rescale)) {
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const float aa = __shfl_sync(kFull, alpha[r], 8 * t);
            const float ab = __shfl_sync(kFull, alpha[r], 8 * t + 4);
#pragma unroll
            for (int i = 0; i < D / 16; ++i) {
                o[r][i][0] *= aa;
                o[r][i][1] *= ab;
                o[r][i][2] *= aa;
                o[r][i][3] *= ab;
            }
        }
    }
}

// Query fragments of a unit: a0/a2 rows 0-7, a1/a3 rows 8-15 (used when NR == 2).
template <int D>
struct QFrag {
    uint32_t a0[D / 16], a1[D / 16], a2[D / 16], a3[D / 16];
    float qm[2];    // power of two the lane's row (g, g + 8) was divided by (E4M3 keys)
};

// Scores q.K of the 16 tokens of one bf16 tile: sc[0] tokens 0-7, sc[1]
// tokens 8-15 (C fragments: row = query row, column = token).
template <int D, int NR>
__device__ __forceinline__ void scores_bf16(uint32_t kbase, const QFrag<D>& qf, float (&sc)[2][4],
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
        const uint32_t a1 = NR == 2 ? qf.a1[s] : 0u, a3 = NR == 2 ? qf.a3[s] : 0u;
        mma_bf16(sc[0], qf.a0[s], a1, qf.a2[s], a3, r[0], r[1]);
        mma_bf16(sc[1], qf.a0[s], a1, qf.a2[s], a3, r[2], r[3]);
    }
}

// O^T += V^T P^T for one bf16 tile and NR row tiles; P is split into bf16
// hi + lo parts.
template <int D, int NR>
__device__ __forceinline__ void pv_bf16(uint32_t vbase, int nvalid, const float (&pr)[NR][4],
                                        float (&o)[NR][D / 16][4], int lane)
{
    using G = Geom<D, false>;
    const int t = lane & 3;
    const int mi = lane >> 3, ri = lane & 7;
    const int tok = ri + 8 * (mi >> 1);
    const int csel = mi & 1;
    uint32_t h0[NR], h1[NR], e0[NR], e1[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        h0[r] = pack_bf16x2(pr[r][0], pr[r][1]);
        h1[r] = pack_bf16x2(pr[r][2], pr[r][3]);
        e0[r] = pack_bf16x2(pr[r][0] - bf16_lo(h0[r]), pr[r][1] - bf16_hi(h0[r]));
        e1[r] = pack_bf16x2(pr[r][2] - bf16_lo(h1[r]), pr[r][3] - bf16_hi(h1[r]));
    }
    uint32_t m01 = 0xffffffffu, m23 = 0xffffffffu;
    if (nvalid < kBlock) {      // zero V rows past the context (they may hold anything)
        const int t0 = 2 * t;
        m01 = (t0 < nvalid ? 0x0000ffffu : 0u) | (t0 + 1 < nvalid ? 0xffff0000u : 0u);
        m23 = (t0 + 8 < nvalid ? 0x0000ffffu : 0u) | (t0 + 9 < nvalid ? 0xffff0000u : 0u);
    }
#pragma unroll
    for (int i = 0; i < G::MTILES; ++i) {
        uint32_t r4[4];
        ldsm_x4_trans(r4, vbase + tile_off<G>(tok, 2 * i + csel));
        r4[0] &= m01; r4[1] &= m01; r4[2] &= m23; r4[3] &= m23;
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            mma_bf16(o[r][i], r4[0], r4[1], r4[2], r4[3], h0[r], h1[r]);
            mma_bf16(o[r][i], r4[0], r4[1], r4[2], r4[3], e0[r], e1[r]);
        }
    }
}

// Scores of one E4M3 tile: bytes via ldmatrix, widened to f16 in registers.
template <int D, int NR>
__device__ __forceinline__ void scores_fp8(uint32_t kbase, const QFrag<D>& qf, float (&sc)[2][4],
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
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            const int k = c + cc;
            const uint32_t a1 = NR == 2 ? qf.a1[k] : 0u, a3 = NR == 2 ? qf.a3[k] : 0u;
            mma_f16(sc[0], qf.a0[k], a1, qf.a2[k], a3, b[2 * cc][0], b[2 * cc][1]);
            mma_f16(sc[1], qf.a0[k], a1, qf.a2[k], a3, b[2 * cc + 1][0], b[2 * cc + 1][1]);
        }
    }
}

// O^T += V^T P^T for one E4M3 tile and NR row tiles; P in f16.
template <int D, int NR>
__device__ __forceinline__ void pv_fp8(uint32_t vbase, int nvalid, const float (&pr)[NR][4],
                                       float (&o)[NR][D / 16][4], int lane)
{
    using G = Geom<D, true>;
    const int g = lane >> 2, t = lane & 3;
    uint32_t pf0[NR], pf1[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        pf0[r] = pack_f16x2(pr[r][0], pr[r][1]);
        pf1[r] = pack_f16x2(pr[r][2], pr[r][3]);
    }
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
#pragma unroll
            for (int r = 0; r < NR; ++r)
                mma_f16(o[r][2 * w + e], a[0], a[1], a[2], a[3], pf0[r], pf1[r]);
        }
    }
}

// NBK consecutive tiles of one stream (K at kb[j], V right after it), NR row
// tiles: scores of every tile first, one softmax update over all of them,
// then P.V.
template <int D, bool FP8, int NBK, int NR>
__device__ __forceinline__ void attend_tiles(const uint32_t (&kb)[NBK], int nvalid_last,
                                             const QFrag<D>& qf, const float (&sl2)[NR],
                                             float (&m)[NR], float (&l)[NR],
                                             float (&o)[NR][D / 16][4], int lane)
{
    using G = Geom<D, FP8>;
    float sc[NBK][2][4];
#pragma unroll
    for (int j = 0; j < NBK; ++j) {
        if (FP8) scores_fp8<D, NR>(kb[j], qf, sc[j], lane);
        else scores_bf16<D, NR>(kb[j], qf, sc[j], lane);
    }
    float pr[NBK][NR][4];
    softmax_update<D, NBK, NR>(sc, nvalid_last, sl2, m, l, o, pr, lane);
#pragma unroll
    for (int j = 0; j < NBK; ++j) {
        const int nv = j == NBK - 1 ? nvalid_last : kBlock;
        if (FP8) pv_fp8<D, NR>(kb[j] + G::TILE, nv, pr[j], o, lane);
        else pv_bf16<D, NR>(kb[j] + G::TILE, nv, pr[j], o, lane);
    }
}

// The same, for a kernel holding NRK >= 1 row tiles of state of which the
// stream uses nr (1 or NRK).
template <int D, bool FP8, int NBK, int NRK>
__device__ __forceinline__ void attend(int nr, const uint32_t (&kb)[NBK], int nvalid_last,
                                       const QFrag<D>& qf, const float (&sl2)[NRK],
                                       float (&m)[NRK], float (&l)[NRK],
                                       float (&o)[NRK][D / 16][4], int lane)
{
    if constexpr (NRK == 2) {
        if (nr == 2) {
            attend_tiles<D, FP8, NBK, 2>(kb, nvalid_last, qf, sl2, m, l, o, lane);
            return;
        }
    }
    attend_tiles<D, FP8, NBK, 1>(kb, nvalid_last, qf,
                                 *reinterpret_cast<const float(*)[1]>(&sl2[0]),
                                 *reinterpret_cast<float(*)[1]>(&m[0]),
                                 *reinterpret_cast<float(*)[1]>(&l[0]),
                                 *reinterpret_cast<float(*)[1][D / 16][4]>(&o[0]), lane);
}

// Query fragment rows of one query head (head index within sequence s);
// `live` false gives a zero row.  bf16 keys: a holds elements (16k + 2t,
// 16k + 2t + 1), b elements (16k + 8 + 2t, ...); E4M3 keys (f16 operands):
// the four consecutive elements 16k + 4t .. 16k + 4t + 3, in the order
// the byte-wise key fragments use.
//
// f16 holds every bfloat16 value of magnitude 2^-14 .. 65504 exactly but
// overflows above 65504, so for E4M3 keys a row whose largest |element| is
// 2^15 or more is first divided by a power of two 2^e that brings it into
// [2^14, 2^15) (exact), and 2^e is returned so that the row's scores are
// multiplied by it again with the softmax scale.  Elements below 2^-24 of the
// (divided) row round to zero in f16: they change a score by less than
// D * 2^-25 * 448 code units, against a largest term of at least 2^14.
// bf16 keys take the bf16 query as it is (returns 1).
template <int D, bool FP8>
__device__ __forceinline__ float load_q_row(const DecodeParams& p, int s, int head, bool live,
                                            int lane, uint32_t (&a)[D / 16],
                                            uint32_t (&b)[D / 16])
{
    const int t = lane & 3;
    const uint16_t* qh = p.q + ((size_t)(live ? s : 0) * p.Hq + (live ? head : 0)) * D;
    if constexpr (!FP8) {
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
            const uint32_t* q32 = reinterpret_cast<const uint32_t*>(qh);
            a[k] = live ? __ldg(q32 + 8 * k + t) : 0u;
            b[k] = live ? __ldg(q32 + 8 * k + 4 + t) : 0u;
        }
        return 1.f;
    } else {
        uint2 v[D / 16];
        float amax = 0.f;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
            v[k] = make_uint2(0u, 0u);
            if (live) v[k] = __ldg(reinterpret_cast<const uint2*>(qh + 16 * k + 4 * t));
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16_lo(v[k].x)), fabsf(bf16_hi(v[k].x))),
                                     fmaxf(fabsf(bf16_lo(v[k].y)), fabsf(bf16_hi(v[k].y)))));
        }
        // the row's D elements sit in its 4 lanes (t = 0..3)
        amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
        float down = 1.f, up = 1.f;
        if (amax >= 32768.f) {
            // amax = 1.f * 2^(E - 127) with E its biased exponent; e = E - 141
            // (e <= 113 for a finite amax: both powers are normal floats)
            const int e = (int)((__float_as_uint(amax) >> 23) & 0xffu) - 141;
            down = __uint_as_float((uint32_t)(127 - e) << 23);
            up = __uint_as_float((uint32_t)(127 + e) << 23);
        }
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
            a[k] = pack_f16x2(bf16_lo(v[k].x) * down, bf16_hi(v[k].x) * down);
            b[k] = pack_f16x2(bf16_lo(v[k].y) * down, bf16_hi(v[k].y) * down);
        }
        return up;
    }
}

// Query fragments of a stream: the G heads of KV head h of sequence s, or
// (prefix chunk c) row r = j*G + i is head h*G + i of the chunk's member j.
template <int D, bool FP8, int NR>
__device__ __forceinline__ void load_q(const DecodeParams& p, bool chunk, int sc, int h, int rows,
                                       int lane, QFrag<D>& qf)
{
    const int g = lane >> 2;
    qf.qm[1] = 1.f;
    if (!chunk) {
        qf.qm[0] = load_q_row<D, FP8>(p, sc, h * p.G + g, g < p.G, lane, qf.a0, qf.a2);
        if constexpr (NR == 2)
            qf.qm[1] = load_q_row<D, FP8>(p, sc, h * p.G + g + 8, g + 8 < p.G, lane, qf.a1,
                                          qf.a3);
        return;
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        const int row = g + 8 * r;
        const int j = row / p.G, i = row - j * p.G;
        int s = -1;
        if (row < rows) s = __ldg(p.chunk + (size_t)sc * KV_PREFIX_CHUNK_INTS + 2 + j);
        const bool live = s >= 0 && s < p.B;
        if (r == 0) qf.qm[0] = load_q_row<D, FP8>(p, s, h * p.G + i, live, lane, qf.a0, qf.a2);
        else qf.qm[1] = load_q_row<D, FP8>(p, s, h * p.G + i, live, lane, qf.a1, qf.a3);
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

// The run of units of one (stream, KV head) inside a warp's range.
struct Seg {
    int pair;          // stream * Hkv + h
    int s;             // own stream: the sequence; prefix chunk: the chunk
    int h;
    bool chunk;
    int rows;          // query rows (G, or members * G)
    int nr;            // row tiles in use (1 or 2)
    int base, end;     // the stream's blocks [base, end) of its block-table row
    int first, last;   // the blocks this warp saw
    int i0;            // position of the first of them in the warp's range
    int cj;            // sequence with a shared prefix: (chunk << 4) | member, else -1
};

// End of a segment: write the final output if the warp saw a whole
// sequence stream with no shared prefix, otherwise store a partial (rows of
// the segment, unnormalised, with their (max, sum)) for the merge kernel.
// The warp holding the stream's first block also records which warps hold
// the rest.  Only plain stores: a stream switch in mid-range does not stall
// the warp's pipeline.
template <int D, bool FP8, int NR>
__device__ __forceinline__ void finalize(const DecodeParams& p, int wl, int q, int b0,
                                         int slot_base, const Seg& sg,
                                         const float (&m)[NR], const float (&l)[NR],
                                         const float (&o)[NR][D / 16][4], int lane)
{
    const int g = lane >> 2, t = lane & 3;
    // this warp's partial slot: each team (sub-group) has its own run of
    // slots, in which pair x's partial of the team's warp wl goes to x + wl
    const int hsh = hshift_of<NR>(p);
    const int team = sg.pair & ((1 << hsh) - 1);
    const size_t slot = (size_t)slot_base + (size_t)team * p.team_slots +
                        (size_t)(sg.pair >> hsh) + wl;
    float la[NR], lb[NR], ma[NR], mb[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        float lt = l[r] + __shfl_xor_sync(kFull, l[r], 1);
        lt += __shfl_xor_sync(kFull, lt, 2);
        la[r] = __shfl_sync(kFull, lt, 8 * t);
        lb[r] = __shfl_sync(kFull, lt, 8 * t + 4);
        ma[r] = __shfl_sync(kFull, m[r], 8 * t);
        mb[r] = __shfl_sync(kFull, m[r], 8 * t + 4);
    }
    if (!sg.chunk && sg.base == 0 && sg.first == 0 && sg.last == sg.end - 1) {
        const size_t row = (size_t)sg.s * p.Hq + (size_t)sg.h * p.G;
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            if (r >= sg.nr) break;
            const int ha = 8 * r + 2 * t, hb = ha + 1;
            const float ia = la[r] > 0.f ? p.v_scale / la[r] : 0.f;
            const float ib = lb[r] > 0.f ? p.v_scale / lb[r] : 0.f;
#pragma unroll
            for (int i = 0; i < D / 16; ++i) {
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int d = out_dim<D, FP8>(i, g, half);
                    if (ha < p.G) {
                        const float v = o[r][i][2 * half] * ia;
                        const size_t idx = (row + ha) * D + d;
                        if (p.out_f32) reinterpret_cast<float*>(p.out)[idx] = v;
                        else reinterpret_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16_rn(v);
                    }
                    if (hb < p.G) {
                        const float v = o[r][i][2 * half + 1] * ib;
                        const size_t idx = (row + hb) * D + d;
                        if (p.out_f32) reinterpret_cast<float*>(p.out)[idx] = v;
                        else reinterpret_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16_rn(v);
                    }
                }
            }
        }
    } else {
        float* po = p.part_o + slot * p.prow * D;
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            if (r >= sg.nr) break;
            const int ha = 8 * r + 2 * t, hb = ha + 1;
#pragma unroll
            for (int i = 0; i < D / 16; ++i) {
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int d = out_dim<D, FP8>(i, g, half);
                    if (ha < sg.rows) po[ha * D + d] = o[r][i][2 * half] * p.v_scale;
                    if (hb < sg.rows) po[hb * D + d] = o[r][i][2 * half + 1] * p.v_scale;
                }
            }
            if (g == 0) {
                if (ha < sg.rows) p.part_ml[slot * p.prow + ha] = make_float2(ma[r], la[r]);
                if (hb < sg.rows) p.part_ml[slot * p.prow + hb] = make_float2(mb[r], lb[r]);
            }
        }
    }
    if (sg.first == sg.base && lane == 0) {
        // the stream's first block is here: record the first partial slot
        // and the warps whose ranges meet its blocks
        // [flat_first, flat_first + (end - base))
        const int flat_first = b0 + sg.i0;
        const int w_last = (flat_first + (sg.end - sg.base) - 1) / q;
        p.pair_meta[sg.pair] = make_int4((int)slot, w_last - wl + 1, sg.cj, 0);
    }
}

// The fused append of the step's new token of pair (s, h): position L-1,
// i.e. row (L-1) % 16 of the pair's last block `id`.  Writes the cache in
// global memory and the same bytes into this warp's copy of the tile in
// shared memory (which the bulk copy may have filled before the write).
template <int D, bool FP8, int NR>
__device__ __forceinline__ void append_patch(const DecodeParams& p, int s, int h, int id, int L,
                                             uint32_t kst, uint32_t vst, int lane)
{
    using G = Geom<D, FP8>;
    constexpr int CH = D / 8;              // groups of 8 elements per row
    if (lane < 2 * CH) {
        const bool isv = lane >= CH;
        const int c = isv ? lane - CH : lane;
        const int r = (L - 1) & (kBlock - 1);
        // cache and new tokens are indexed by the physical KV head
        const int Hp = hkv_phys<NR>(p), hp = h >> hshift_of<NR>(p);
        const size_t src = ((size_t)s * Hp + hp) * D + 8 * c;
        const size_t dst = (((size_t)id * Hp + hp) * kBlock + r) * D + 8 * c;
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

template <int D, bool FP8, int NR>
__device__ __forceinline__ void split_body(const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                           const DecodeParams& p)
{
    using G = Geom<D, FP8>;
    constexpr int ST = G::STAGES;
    extern __shared__ uint8_t smem_raw[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int w = blockIdx.x * G::WARPS + warp;
    // Groups cut into 2^hshift sub-groups: the warps form one team per
    // sub-group, and every team partitions the same (sequence, KV head,
    // block) units the same way, so the warps of all teams that read a tile
    // do so at about the same time and the repeats hit L2.
    const int hsh = hshift_of<NR>(p), Hkv_p = hkv_phys<NR>(p);
    const int Wt = p.warps_total >> hsh;
    const int team = w / Wt, wl = w - team * Wt;
    if (team >= (1 << hsh)) return;

    const uint32_t sraw = smem_u32(smem_raw);
    const uint32_t sbase = (sraw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (sbase - sraw);
    const uint32_t stage0 = sbase + (uint32_t)(warp * ST * G::STAGE);
    const uint32_t bar0 = sbase + (uint32_t)(G::BAR_OFF + warp * ST * 8);
    const uint32_t stall_bar = sbase + (uint32_t)(G::STALL_OFF + warp * 8);
    int4* meta = reinterpret_cast<int4*>(gbase + G::META_OFF) + warp * ST;

    if (threadIdx.x == 0) {
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    // let the next kernel on the stream launch now, then wait until the
    // previous one has finished and its writes are visible -- with `early`,
    // only before the first access to q, k_new, the outputs or the workspace
    // (the scan, the block-id windows and the first bulk copies overlap the
    // previous kernel's end)
    pdl_launch_dependents();
    bool waited = false;
    if (!p.early) {
        pdl_wait();
        waited = true;
    }

    if (lane == 0) {
#pragma unroll
        for (int st = 0; st < ST; ++st) mbar_init(bar0 + st * 8, 1);
        if (p.test_stall > 0) mbar_init(stall_bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    int st = 0;                   // the ring carries over from one phase to the next
    uint32_t phase = 0;

    // Phase 0 (NR == 2 kernels with prefix chunks): the chunk streams, cut
    // into equal per-warp ranges; phase 1: the sequence streams, likewise.
    // Every warp takes its share of both, so the costlier chunk units do not
    // pile up on a few warps.
    for (int ph = (NR == 2 && p.nc > 0) ? 0 : 1; ph < 2; ++ph) {
        const int nc = NR == 2 ? p.nc : 0;
        const int s_lo = ph == 0 ? 0 : nc;
        const int ns = ph == 0 ? nc : nc + p.B;           // streams [s_lo, ns)
        const int min_q = ph == 0 ? kMinBlocksPerWarpChunk : p.min_q1;
        const int slot_base = ph == 0 ? 0 : p.slot_base;

        // ---- 1. total work and this warp's range --------------------------------
        constexpr int U = 8;           // first 256 streams stay in registers
        int nbv[U], incl[U];
        int carry = 0;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int sg = s_lo + u * 32 + lane;
            nbv[u] = sg < ns ? max(stream_at<NR>(p, sg).nblk, 0) : 0;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            incl[u] = warp_incl_scan(nbv[u] * Hkv_p, lane) + carry;
            carry = __shfl_sync(kFull, incl[u], 31);
        }
        int total = carry;
        // streams past the first 256: 256 at a time, all loads issued together
        for (int base = s_lo + U * 32; base < ns; base += U * 32) {
            int v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int sg = base + u * 32 + lane;
                v[u] = sg < ns ? max(stream_at<NR>(p, sg).nblk, 0) : 0;
            }
            int sum = 0;
#pragma unroll
            for (int u = 0; u < U; ++u) sum += v[u];
            total += warp_sum(sum) * Hkv_p;
        }
        if (total == 0) continue;
        int q = (total + Wt - 1) / Wt;
        if (q < min_q) q = min_q;
        const int weff = (total + q - 1) / q;
        if (wl >= weff) continue;
        const int b0 = wl * q;
        const int cnt = min(q, total - b0);

        // ---- 2. the (stream, head, block) where the range starts ----------------
        int s0 = -1, excl = 0;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const unsigned mball = __ballot_sync(kFull, incl[u] > b0);
            if (s0 < 0 && mball) {
                const int src = __ffs(mball) - 1;
                s0 = s_lo + u * 32 + src;
                excl = __shfl_sync(kFull, incl[u] - nbv[u] * Hkv_p, src);
            }
        }
        if (s0 < 0) {
            int c2 = carry;
            for (int base = s_lo + U * 32; base < ns && s0 < 0; base += U * 32) {
                int v[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int sg = base + u * 32 + lane;
                    v[u] = sg < ns ? max(stream_at<NR>(p, sg).nblk, 0) * Hkv_p : 0;
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
        if (s0 < 0) continue;      // unreachable with consistent input
        const Stream S0 = stream_at<NR>(p, s0);
        if (S0.nblk <= 0) continue;     // inputs changed under the launch
        const int off0 = b0 - excl;
        const int h0 = off0 / S0.nblk;
        const int j0 = off0 - h0 * S0.nblk;

        // ---- 3. block-id windows and the copy issue -------------------------------
        Win cur, nxt;
        int wb = 0;
        fill_window<NR>(cur, p, ns, s0, h0, j0, S0, 0, cnt, lane);
        nxt = cur;
        auto refill_next = [&](int pos0) {
            const int cs = __shfl_sync(kFull, cur.s, 31), ch = __shfl_sync(kFull, cur.h, 31);
            const int cb = __shfl_sync(kFull, cur.blk, 31) + 1;
            // the stream of the window's last entry, from registers (no loads)
            Stream S;
            S.L = __shfl_sync(kFull, cur.L, 31);
            S.base = NR == 2 ? __shfl_sync(kFull, cur.base, 31) : 0;
            S.row = NR == 2 ? __shfl_sync(kFull, cur.row, 31) : cs;
            S.nblk = (S.L + kBlock - 1) / kBlock - S.base;
            S.cj = -1;
            fill_window<NR>(nxt, p, ns, cs, ch, cb - S.base, S, pos0, cnt, lane);
        };
        if (cnt > 32) refill_next(32);

        // unit j (of this phase's range) into ring stage `sst`
        auto issue = [&](int j, int sst) {
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
                const int pair = s * p.Hkv + (h << hsh) + team;
                meta[sst] = make_int4(valid ? pair : -1 - pair, blk, L, id);
                const uint32_t bar = bar0 + sst * 8;
                const uint32_t dst = stage0 + (uint32_t)(sst * G::STAGE);
                if (valid) {
                    fence_proxy_async_smem();
                    mbar_arrive_expect_tx(bar, (uint32_t)G::STAGE);
                    const int z = id * Hkv_p + h;
                    // KV tiles are read once per step: keep them from evicting
                    // the block tables, queries and partials from L2
                    const uint64_t pol = l2_evict_first_policy();
#pragma unroll
                    for (int b = 0; b < G::NBOX; ++b)
                        tma_load_3d_hint(dst + b * G::BOXB, &tm_k, b * (G::BOXW / G::ES), 0, z,
                                         bar, pol);
#pragma unroll
                    for (int b = 0; b < G::NBOX; ++b)
                        tma_load_3d_hint(dst + G::TILE + b * G::BOXB, &tm_v,
                                         b * (G::BOXW / G::ES), 0, z, bar, pol);
                } else {
                    raise_flag(&g_decode_err, KV_DEVERR_BLOCK_OUT_OF_RANGE, id);
                    mbar_arrive(bar);
                }
            }
        };

        {
            int sst = st;
            const int npro = min(ST, cnt);
            for (int j = 0; j < npro; ++j) {
                issue(j, sst);
                if (++sst == ST) sst = 0;
            }
        }

        if (!waited) {
            pdl_wait();
            waited = true;
        }
        // ---- 4. main loop ------------------------------------------------------------
        // Two consecutive tiles of a sequence stream are consumed together
        // where the range allows: one softmax update and one loop turn per 32
        // tokens.  (Prefix chunk segments take one tile per update: a second
        // inlined copy of their two-row-tile math costs more than it saves.)
        QFrag<D> qf;
        float sl2r[NR];           // score scale of the lane's rows (g, g + 8)
        float o[NR][D / 16][4];
        float m[NR], l[NR];
        Seg sg;
        sg.pair = -1;
        bool open = false;
        // Wait for unit i in stage `sst`; on time-out flag the error and let the
        // copies of units [i, issued_end) land before the warp gives up.
        auto give_up = [&](int i, int sst, uint32_t phs, int issued_end) {
            if (lane == 0) {
                raise_flag(&g_decode_err, KV_DEVERR_PIPELINE_TIMEOUT, i);
                for (int j = i; j < issued_end; ++j) {
                    mbar_wait_bounded(bar0 + sst * 8, phs, kWaitLimit);
                    if (++sst == ST) { sst = 0; phs ^= 1u; }
                }
            }
            __syncwarp();
        };
        auto wait_unit = [&](int i, int sst, uint32_t phs, int issued_end) -> bool {
            const bool ok = __all_sync(kFull, mbar_wait_bounded(bar0 + sst * 8, phs, kWaitLimit));
            if (!ok) give_up(i, sst, phs, issued_end);
            return ok;
        };
        // Test hook: a first wait on a barrier that nothing arrives on, for
        // test_stall clocks; the copies issued so far are still waited for,
        // on their own barriers, at the full limit.
        if (p.test_stall > 0 &&
            !__all_sync(kFull, mbar_wait_bounded(stall_bar, 0u, p.test_stall))) {
            give_up(0, st, phase, min(cnt, ST));
            return;
        }
        for (int i = 0; i < cnt;) {
            const int issued_end = min(cnt, i + ST);
            if (!wait_unit(i, st, phase, issued_end)) return;
            const int4 mt = meta[st];
            const bool valid = mt.x >= 0;
            const int pair = valid ? mt.x : -1 - mt.x;
            const int blk = mt.y, L = mt.z;
            if (pair != sg.pair) {
                if (open) finalize<D, FP8, NR>(p, wl, q, b0, slot_base, sg, m, l, o, lane);
                open = true;
                const int sig = pair / p.Hkv;
                const Stream S = stream_at<NR>(p, sig);
                sg.pair = pair;
                sg.h = pair - sig * p.Hkv;
                sg.chunk = NR == 2 && sig < nc;
                sg.s = sg.chunk ? sig : sig - nc;
                sg.rows = p.G;
                if (sg.chunk)
                    sg.rows = p.G * __ldg(p.chunk + (size_t)sig * KV_PREFIX_CHUNK_INTS + 1);
                sg.nr = NR == 2 && sg.rows > 8 ? 2 : 1;
                sg.base = S.base;
                sg.end = S.base + S.nblk;
                sg.cj = S.cj;
                sg.first = blk;
                sg.i0 = i;
                load_q<D, FP8, NR>(p, sg.chunk, sg.s, sg.h, sg.rows, lane, qf);
#pragma unroll
                for (int r = 0; r < NR; ++r) sl2r[r] = FP8 ? p.sl2 * qf.qm[r] : p.sl2;
#pragma unroll
                for (int r = 0; r < NR; ++r) {
                    m[r] = -INFINITY;
                    l[r] = 0.f;
#pragma unroll
                    for (int a = 0; a < D / 16; ++a)
                        o[r][a][0] = o[r][a][1] = o[r][a][2] = o[r][a][3] = 0.f;
                }
            }
            const int st2 = st + 1 == ST ? 0 : st + 1;
            const uint32_t phase2 = st + 1 == ST ? phase ^ 1u : phase;
            bool two = false;
            if (!sg.chunk && valid && i + 1 < cnt) {
                __syncwarp();            // unit i+1's metadata was written by lane 0
                two = meta[st2].x == mt.x;
            }
            const uint32_t kb = stage0 + (uint32_t)(st * G::STAGE);
            // the fused append writes the new token into its sequence's last block
            const bool own_last = !sg.chunk && p.k_new != nullptr;
            if (two) {
                if (!wait_unit(i + 1, st2, phase2, issued_end)) return;
                const int id2 = meta[st2].w;
                const uint32_t kb2 = stage0 + (uint32_t)(st2 * G::STAGE);
                const int rest = L - (blk + 1) * kBlock;
                const int nvalid = min(kBlock, rest);
                if (own_last && nvalid == rest)
                    append_patch<D, FP8, NR>(p, sg.s, sg.h, id2, L, kb2, kb2 + G::TILE, lane);
                const uint32_t kbs[2] = {kb, kb2};
                attend<D, FP8, 2, NR>(sg.nr, kbs, nvalid, qf, sl2r, m, l, o, lane);
                sg.last = blk + 1;
                __syncwarp();
                if (i + ST < cnt) issue(i + ST, st);
                if (i + 1 + ST < cnt) issue(i + 1 + ST, st2);
                st = st2 + 1 == ST ? 0 : st2 + 1;
                phase = st2 + 1 == ST ? phase2 ^ 1u : phase2;
                i += 2;
            } else {
                sg.last = blk;
                if (valid) {
                    const int nvalid = min(kBlock, L - blk * kBlock);
                    if (own_last && nvalid == L - blk * kBlock)
                        append_patch<D, FP8, NR>(p, sg.s, sg.h, mt.w, L, kb, kb + G::TILE, lane);
                    const uint32_t kbs[1] = {kb};
                    attend<D, FP8, 1, NR>(sg.nr, kbs, nvalid, qf, sl2r, m, l, o, lane);
                }
                __syncwarp();
                if (i + ST < cnt) issue(i + ST, st);
                st = st2;
                phase = phase2;
                i += 1;
            }
        }
        if (open) finalize<D, FP8, NR>(p, wl, q, b0, slot_base, sg, m, l, o, lane);
    }
}

// Plain decoding: one row tile per unit.
template <int D, bool FP8>
__global__ void __launch_bounds__(Geom<D, FP8>::WARPS * 32, Geom<D, FP8>::MIN_CTAS)
paged_decode_split_kernel(const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const DecodeParams p)
{
    split_body<D, FP8, 1>(tm_k, tm_v, p);
}

// Shared-prefix decoding: prefix chunks with up to 16 query rows, then the
// sequences.
template <int D, bool FP8>
__global__ void __launch_bounds__(Geom<D, FP8>::WARPS * 32, Geom<D, FP8>::MIN_CTAS)
paged_decode_prefix_kernel(const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v, const DecodeParams p)
{
    split_body<D, FP8, 2>(tm_k, tm_v, p);
}

// -------------------------------------------------------------------- merge

struct MergeParams {
    void* out;
    const int32_t* ctx;
    const float* part_o;
    const float2* part_ml;
    const int4* pair_meta;
    const int32_t* chunk;    // prefix chunks (checked here, read by the split kernel)
    const int32_t* seq_chunk;
    int nc;
    int B, Hq, Hkv, G, max_blocks;
    int prow;                // rows per partial slot
    int nslots;              // partial slots in the workspace
    int out_f32;
    int early;               // context lengths are stable inputs: read them before the wait
};

// One CTA per (sequence, KV head): merge the partials the split kernel left
// for it -- those of its own blocks and, with a shared prefix, its rows of
// the prefix chunk's partials -- (a sequence seen whole by one warp was
// written there already), or write zeros for an empty context.  Thread t
// owns output float4 column t of the pair's G x D block; the (max, sum)
// terms of up to 64 partials at a time go through shared memory, and a
// thread's partial loads are independent of one another, so the merge costs
// a few L2 round trips.
constexpr int kMergeMaxThreads = 512;   // >= 16 rows x 128 / 4 columns
constexpr int kMergeRows = 16;          // query rows of a pair at most
constexpr int kMergeChunk = 64;
constexpr int kMergeDirect = 8;      // up to this many partials: no staging

// Threads of a merge CTA: one per float4 column of the G x D block, whole warps.
inline int merge_threads(int G, int D) { return (G * D / 4 + 31) / 32 * 32; }

// Small CTAs with few registers, so that they fit beside the split kernel's
// CTAs and start (programmatic dependent launch) before it drains.
template <int D>
__global__ void __launch_bounds__(kMergeMaxThreads, 2) paged_decode_merge_kernel(const MergeParams p)
{
    __shared__ float2 sml[kMergeChunk * kMergeRows];
    const int s = blockIdx.x / p.Hkv, h = blockIdx.x - s * p.Hkv;
    const int t = threadIdx.x;
    const int nthr = blockDim.x;
    const int cols = p.G * (D / 4);
    const size_t row = (size_t)s * p.Hq + (size_t)h * p.G;
    // with early inputs the length is read while the split kernel drains
    int L = 0;
    if (p.early) seq_blocks(p.ctx, s, p.max_blocks, L, true);
    // the next kernel may start only once the split kernel (and with it the
    // step's appends to the cache) is complete: a following call that reads
    // its inputs early sees them
    pdl_wait();
    pdl_launch_dependents();
    if (!p.early) seq_blocks(p.ctx, s, p.max_blocks, L, true);
    if (p.nc > 0 && h == 0 && t == 0) {
        // report inconsistent prefix-chunk entries (the split kernel only reads)
        int c, j, lead, members;
        prefix_of(p.chunk, p.seq_chunk, p.nc, p.B, p.G, p.max_blocks, s, L, c, j, true);
        if (s < p.nc) chunk_blocks(p.chunk, s, p.B, p.G, p.max_blocks, lead, members, true);
    }
    if (L <= 0) {
        if (t < cols) store4(p, row * D + 4 * t, 0.f, 0.f, 0.f, 0.f);
        return;
    }
    const int pair = (p.nc + s) * p.Hkv + h;
    const int4 mt = p.pair_meta[pair];
    const int na = mt.y;
    // the table is rewritten by every split launch; refuse anything that
    // would leave the workspace (only an aborted split launch leaves it stale)
    if (mt.x < 0 || na < 1 || (long long)mt.x + na > (long long)p.nslots) return;
    // the prefix chunk's partials (recorded by the split kernel): slots from
    // cpair + w0, rows from member * G
    int nb = 0, crow = 0;
    long long cslot0 = 0;
    if (mt.z >= 0 && (mt.z >> 4) < p.nc) {
        const int cpair = (mt.z >> 4) * p.Hkv + h;
        const int4 cm = p.pair_meta[cpair];
        if (cm.x < 0 || cm.y < 1 || (long long)cm.x + cm.y > (long long)p.nslots ||
            (mt.z & 15) * p.G + p.G > p.prow)
            return;
        nb = cm.y;
        cslot0 = cm.x;
        crow = (mt.z & 15) * p.G;
    }
    if (na <= 1 && nb == 0) return;
    const long long aslot0 = mt.x;
    const int n = na + nb;
    const int g = t / (D / 4), d4 = t % (D / 4);
    const bool live = t < cols;
    // partial k: its row of (max, sum) and its float4 column of the output
    auto prow_of = [&](int k) -> size_t {
        return k < na ? (size_t)(aslot0 + k) * p.prow + g
                      : (size_t)(cslot0 + (k - na)) * p.prow + crow + g;
    };
    if (n <= kMergeDirect) {
        // few partials: every load at once (one round trip), same arithmetic
        // and order as the staged path below
        if (!live) return;
        float2 v[kMergeDirect];
        float4 ov[kMergeDirect];
#pragma unroll
        for (int k = 0; k < kMergeDirect; ++k) {
            if (k < n) {
                const size_t r = prow_of(k);
                v[k] = __ldcg(&p.part_ml[r]);
                ov[k] = __ldcg(reinterpret_cast<const float4*>(p.part_o + r * D) + d4);
            }
        }
        float M = -INFINITY;
#pragma unroll
        for (int k = 0; k < kMergeDirect; ++k)
            if (k < n && v[k].y > 0.f) M = fmaxf(M, v[k].x);
        float den = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < kMergeDirect; ++k) {
            if (k < n) {
                const float f = v[k].y > 0.f ? exp2f(v[k].x - M) : 0.f;
                den += f * v[k].y;
                acc.x += f * ov[k].x;
                acc.y += f * ov[k].y;
                acc.z += f * ov[k].z;
                acc.w += f * ov[k].w;
            }
        }
        const float inv = den > 0.f ? 1.f / den : 0.f;
        store4(p, (row + g) * D + 4 * d4, acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        return;
    }
    float M = -INFINITY, den = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k0 = 0; k0 < n; k0 += kMergeChunk) {
        const int nk = min(kMergeChunk, n - k0);
        __syncthreads();
        for (int i = t; i < nk * p.G; i += nthr) {
            const int kk = i / p.G, gg = i - kk * p.G;
            const int k = k0 + kk;
            const size_t r = k < na ? (size_t)(aslot0 + k) * p.prow + gg
                                    : (size_t)(cslot0 + (k - na)) * p.prow + crow + gg;
            float2 v = __ldcg(&p.part_ml[r]);
            if (!(v.y > 0.f)) v = make_float2(-INFINITY, 0.f);     // empty partial
            sml[kk * kMergeRows + gg] = v;
        }
        __syncthreads();
        if (!live) continue;
        float cm = -INFINITY;
        for (int k = 0; k < nk; ++k) cm = fmaxf(cm, sml[k * kMergeRows + g].x);
        const float Mn = fmaxf(M, cm);
        const float r = Mn == -INFINITY ? 0.f : exp2f(M - Mn);
        den *= r;
        acc.x *= r; acc.y *= r; acc.z *= r; acc.w *= r;
        M = Mn;
#pragma unroll 4
        for (int kk = 0; kk < nk; ++kk) {
            const int k = k0 + kk;
            const size_t prw = k < na ? (size_t)(aslot0 + k) * p.prow + g
                                      : (size_t)(cslot0 + (k - na)) * p.prow + crow + g;
            const float4 o = __ldcg(reinterpret_cast<const float4*>(p.part_o + prw * D) + d4);
            const float2 v = sml[kk * kMergeRows + g];
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

// One CTA per (sequence, KV head, query row): the row's partials are split
// over the CTA's warps (warp w takes partials w, w + W, ...), each lane one
// float4 column; every warp combines its partials with the running
// (max, sum) rule, loading kMergeRowBatch of them at once, and the warps'
// results are combined through shared memory.  Many partials per pair
// (long contexts, wide groups) cost a few round trips instead of one per
// few partials, and rows of one pair run on different SMs.
constexpr int kMergeRowWarps = 4;
constexpr int kMergeRowBatch = 4;

template <int D>
__global__ void __launch_bounds__(kMergeRowWarps * 32) paged_decode_merge_row_kernel(const MergeParams p)
{
    static_assert(D / 4 <= 32, "one float4 column per lane");
    __shared__ float sM[kMergeRowWarps][32], sDen[kMergeRowWarps][32];
    __shared__ float4 sAcc[kMergeRowWarps][32];
    const int row_g = blockIdx.x % p.G;
    const int ph = blockIdx.x / p.G;
    const int s = ph / p.Hkv, h = ph - s * p.Hkv;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const bool live = lane < D / 4;
    const size_t row = (size_t)s * p.Hq + (size_t)h * p.G + row_g;
    int L = 0;
    if (p.early) seq_blocks(p.ctx, s, p.max_blocks, L, row_g == 0 && t == 0);
    pdl_wait();
    pdl_launch_dependents();
    if (!p.early) seq_blocks(p.ctx, s, p.max_blocks, L, row_g == 0 && t == 0);
    if (p.nc > 0 && h == 0 && row_g == 0 && t == 0) {
        int c, j, lead, members;
        prefix_of(p.chunk, p.seq_chunk, p.nc, p.B, p.G, p.max_blocks, s, L, c, j, true);
        if (s < p.nc) chunk_blocks(p.chunk, s, p.B, p.G, p.max_blocks, lead, members, true);
    }
    if (L <= 0) {
        if (warp == 0 && live) store4(p, row * D + 4 * lane, 0.f, 0.f, 0.f, 0.f);
        return;
    }
    const int pair = (p.nc + s) * p.Hkv + h;
    const int4 mt = p.pair_meta[pair];
    const int na = mt.y;
    if (mt.x < 0 || na < 1 || (long long)mt.x + na > (long long)p.nslots) return;
    int nb = 0, crow = 0;
    long long cslot0 = 0;
    if (mt.z >= 0 && (mt.z >> 4) < p.nc) {
        const int cpair = (mt.z >> 4) * p.Hkv + h;
        const int4 cm = p.pair_meta[cpair];
        if (cm.x < 0 || cm.y < 1 || (long long)cm.x + cm.y > (long long)p.nslots ||
            (mt.z & 15) * p.G + p.G > p.prow)
            return;
        nb = cm.y;
        cslot0 = cm.x;
        crow = (mt.z & 15) * p.G;
    }
    if (na <= 1 && nb == 0) return;
    const long long aslot0 = mt.x;
    const int n = na + nb;
    auto prow_of = [&](int k) -> size_t {
        return k < na ? (size_t)(aslot0 + k) * p.prow + row_g
                      : (size_t)(cslot0 + (k - na)) * p.prow + crow + row_g;
    };
    float M = -INFINITY, den = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k0 = warp; k0 < n; k0 += kMergeRowWarps * kMergeRowBatch) {
        float2 v[kMergeRowBatch];
        float4 ov[kMergeRowBatch];
#pragma unroll
        for (int e = 0; e < kMergeRowBatch; ++e) {
            const int k = k0 + e * kMergeRowWarps;
            if (k < n) {
                const size_t r = prow_of(k);
                v[e] = __ldcg(&p.part_ml[r]);
                if (live) ov[e] = __ldcg(reinterpret_cast<const float4*>(p.part_o + r * D) + lane);
            }
        }
        float bm = M;
#pragma unroll
        for (int e = 0; e < kMergeRowBatch; ++e)
            if (k0 + e * kMergeRowWarps < n && v[e].y > 0.f) bm = fmaxf(bm, v[e].x);
        const float rr = bm == -INFINITY ? 0.f : exp2f(M - bm);
        den *= rr;
        acc.x *= rr; acc.y *= rr; acc.z *= rr; acc.w *= rr;
        M = bm;
#pragma unroll
        for (int e = 0; e < kMergeRowBatch; ++e) {
            if (k0 + e * kMergeRowWarps < n && v[e].y > 0.f) {
                const float f = exp2f(v[e].x - M);
                den += f * v[e].y;
                if (live) {
                    acc.x += f * ov[e].x;
                    acc.y += f * ov[e].y;
                    acc.z += f * ov[e].z;
                    acc.w += f * ov[e].w;
                }
            }
        }
    }
    sM[warp][lane] = M;
    sDen[warp][lane] = den;
    sAcc[warp][lane] = acc;
    __syncthreads();
    if (warp != 0 || !live) return;
    float Mt = -INFINITY;
#pragma unroll
    for (int w = 0; w < kMergeRowWarps; ++w) Mt = fmaxf(Mt, sM[w][lane]);
    float dt = 0.f;
    float4 at = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kMergeRowWarps; ++w) {
        const float f = sM[w][lane] == -INFINITY ? 0.f : exp2f(sM[w][lane] - Mt);
        dt += f * sDen[w][lane];
        const float4 a = sAcc[w][lane];
        at.x += f * a.x; at.y += f * a.y; at.z += f * a.z; at.w += f * a.w;
    }
    const float inv = dt > 0.f ? 1.f / dt : 0.f;
    store4(p, row * D + 4 * lane, at.x * inv, at.y * inv, at.z * inv, at.w * inv);
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
    VariantInfo v[2][2][2];    // [D==128][fp8][NR==2]
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
std::atomic<long long> g_test_stall{0};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

template <int D, bool FP8, int NR>
const void* split_fn()
{
    if constexpr (NR == 2) return reinterpret_cast<const void*>(&paged_decode_prefix_kernel<D, FP8>);
    return reinterpret_cast<const void*>(&paged_decode_split_kernel<D, FP8>);
}

template <int D, bool FP8, int NR>
int variant_setup(VariantInfo& vi)
{
    using G = Geom<D, FP8>;
    const void* fn = split_fn<D, FP8, NR>();
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM) !=
        cudaSuccess)
        return KV_ERR_CUDA;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, G::WARPS * 32, G::SMEM) !=
            cudaSuccess ||
        n <= 0)
        return KV_ERR_CUDA;
    vi.ctas_per_sm = n;
    vi.ready = true;
    return KV_OK;
}

template <int D, bool FP8>
int variant_setup_nr(VariantInfo& vi, int nr)
{
    return nr == 2 ? variant_setup<D, FP8, 2>(vi) : variant_setup<D, FP8, 1>(vi);
}

int warps_per_cta(int D, bool fp8)
{
    if (D == 128) return fp8 ? Geom<128, true>::WARPS : Geom<128, false>::WARPS;
    return fp8 ? Geom<64, true>::WARPS : Geom<64, false>::WARPS;
}

// Device facts and per-variant occupancy, cached per device.
int device_info(int D, bool fp8, int nr, int& sms, int& ctas_per_sm)
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
    VariantInfo& vi = di.v[D == 128][fp8][nr == 2];
    if (!vi.ready) {
        int rc;
        if (D == 128)
            rc = fp8 ? variant_setup_nr<128, true>(vi, nr) : variant_setup_nr<128, false>(vi, nr);
        else
            rc = fp8 ? variant_setup_nr<64, true>(vi, nr) : variant_setup_nr<64, false>(vi, nr);
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
// A tensor map is a pure function of (base address, head dim, element type,
// blocks, KV heads), so the last few are kept: a decode loop calls with the
// same caches every step and skips the encode.  (Virtual addresses are
// unique across the devices of a process.)
struct MapEntry {
    const void* base;
    int D, fp8, num_blocks, Hkv;
    CUtensorMap map;
};
constexpr int kMapCache = 8;
MapEntry g_maps[kMapCache];
int g_map_count = 0, g_map_next = 0;
std::mutex g_map_mu;

int encode_cache_map(CUtensorMap* map, const void* base, int D, bool fp8, int num_blocks,
                     int Hkv);

int make_cache_map(CUtensorMap* map, const void* base, int D, bool fp8, int num_blocks, int Hkv)
{
    std::lock_guard<std::mutex> lk(g_map_mu);
    for (int i = 0; i < g_map_count; ++i) {
        const MapEntry& e = g_maps[i];
        if (e.base == base && e.D == D && e.fp8 == (int)fp8 && e.num_blocks == num_blocks &&
            e.Hkv == Hkv) {
            *map = e.map;
            return KV_OK;
        }
    }
    if (int rc = encode_cache_map(map, base, D, fp8, num_blocks, Hkv)) return rc;
    MapEntry& e = g_maps[g_map_next];
    e.base = base;
    e.D = D;
    e.fp8 = (int)fp8;
    e.num_blocks = num_blocks;
    e.Hkv = Hkv;
    e.map = *map;
    g_map_next = (g_map_next + 1) % kMapCache;
    if (g_map_count < kMapCache) ++g_map_count;
    return KV_OK;
}

int encode_cache_map(CUtensorMap* map, const void* base, int D, bool fp8, int num_blocks, int Hkv)
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

// Partial slots: one per (stream, KV head) plus one per warp (a warp's
// partial of pair x goes to slot x + w).  nr == 2 (prefix chunks, or groups
// of 9-16 rows) gives slots of KV_PREFIX_MAX_ROWS rows, otherwise G rows.
// Hkv is the number of (virtual) KV heads the kernels iterate over.
WsLayout ws_layout(int B, int nc, int Hq, int Hkv, int D, int warps_total, int nr)
{
    const int prow = nr == 2 ? KV_PREFIX_MAX_ROWS : Hq / Hkv;
    const size_t pairs = ((size_t)B + (size_t)nc) * Hkv;
    const size_t slots = pairs + (size_t)warps_total;
    WsLayout L;
    L.part_o = 0;
    L.part_ml = align256(slots * prow * D * sizeof(float));
    L.meta = L.part_ml + align256(slots * prow * sizeof(float2));
    L.total = L.meta + align256(pairs * sizeof(int4));
    return L;
}

// Query heads per KV head, G = Hq / Hkv: up to 8 rows run the kernel with one
// row tile of state, 9-16 the one with two; a larger G (MQA on a many-head
// model) is served as 2^k virtual KV heads of G / 2^k <= 16 rows each.  The
// split kernel's warps then form 2^k teams, one per sub-group, that cut the
// same units the same way, so a tile's 2^k reads come at about the same
// time and all but the first hit L2.
struct HeadSplit {
    int Hkv_v, G_v, hshift;
};

int head_split(int Hq, int Hkv, HeadSplit& hs)
{
    const int G = Hq / Hkv;
    int k = 0;
    while ((G >> k) > KV_PREFIX_MAX_ROWS) ++k;
    if (k > 3 || G % (1 << k) != 0) return KV_ERR_UNSUPPORTED;    // G <= 128, even split
    hs.hshift = k;
    hs.G_v = G >> k;
    hs.Hkv_v = Hkv << k;
    return KV_OK;
}

int check_shape(int num_seqs, int Hq, int Hkv, int D, int kv_dtype)
{
    if (num_seqs < 0 || Hq <= 0 || Hkv <= 0) return KV_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return KV_ERR_INVALID_ARG;
    HeadSplit hs;
    if (int rc = head_split(Hq, Hkv, hs)) return rc;
    if (D != 64 && D != 128) return KV_ERR_UNSUPPORTED;
    if (kv_dtype != KV_DTYPE_BF16 && kv_dtype != KV_DTYPE_FP8_E4M3) return KV_ERR_UNSUPPORTED;
    return KV_OK;
}

// Everything about a launch that the workspace size depends on: the head
// split, the kernel (row tiles nr), the persistent grid and the partial
// slots (a second set of per-warp slots for the prefix-chunk phase).
struct LaunchPlan {
    HeadSplit hs;
    bool wide;             // the tensor-memory kernel (groups above 32 rows, see use_wide)
    int nr, grid, warps_total, slot_warps;
    WsLayout ws;
};

// Groups of more than 32 query rows per KV head (four or more sub-groups) on
// a bf16 cache with head_dim 128 run the wide-group kernel (5th-generation
// tensor cores, all rows of a group in one 128-row MMA); it writes its
// partials in the sub-group layout below, so the same merge kernel follows.
// Measured on GB300 (32 sequences x 8193 tokens, one KV head, fused step):
// 128 rows 57.7 us against 108.9 us for the sub-group kernel, 64 rows 47.6
// against 61.5, 48 rows 51.8 against 60.5; at 32 rows and below the sub-group
// kernel is faster (32 rows 38.5 against 41.5 us, 24 rows 37.5 against 44.4;
// 32 rows at 64 x 16385, 8 x 32769 and 128 x 2049 tokens likewise).
constexpr int kWideMinRows = 33;

bool use_wide(int Hq, int Hkv, int D, bool fp8, int nc)
{
    return !fp8 && D == 128 && nc == 0 && Hq / Hkv >= kWideMinRows;
}

int plan_launch(int B, int nc, int Hq, int Hkv, int D, bool fp8, LaunchPlan& lp)
{
    if (int rc = head_split(Hq, Hkv, lp.hs)) return rc;
    // prefix chunks pack at least two members' rows into 16: G <= 8
    if (nc > 0 && 2 * (Hq / Hkv) > KV_PREFIX_MAX_ROWS) return KV_ERR_UNSUPPORTED;
    lp.nr = (nc > 0 || lp.hs.G_v > 8) ? 2 : 1;
    lp.wide = use_wide(Hq, Hkv, D, fp8, nc);
    int sms = 0, cps = 0;
    if (lp.wide) {
        // partial slots of one sub-group: one per (sequence, KV head) plus
        // one per CTA (a CTA's partial of pair x goes to slot x + CTA)
        sms = num_sms_current();
        if (int rc = wide_setup(Hq / Hkv, cps)) return rc;
        lp.grid = sms * cps;
        lp.warps_total = lp.grid;
        lp.slot_warps = lp.grid << lp.hs.hshift;
        lp.ws = ws_layout(B, 0, Hq, lp.hs.Hkv_v, D, lp.slot_warps, 2);
        return KV_OK;
    }
    if (int rc = device_info(D, fp8, lp.nr, sms, cps)) return rc;
    lp.grid = sms * cps;
    lp.warps_total = lp.grid * warps_per_cta(D, fp8);
    lp.slot_warps = nc > 0 ? 2 * lp.warps_total : lp.warps_total;
    lp.ws = ws_layout(B, nc, Hq, lp.hs.Hkv_v, D, lp.slot_warps, lp.nr);
    return KV_OK;
}

// Launch with programmatic stream serialisation: the kernel may start while
// the previous kernel on the stream drains; it waits on the device
// (griddepcontrol.wait) before touching memory (the split kernel with
// KV_DECODE_EARLY_INPUTS: before touching what the previous kernel may write).
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

struct PrefixArgs {
    const int32_t* chunk;
    const int32_t* seq_chunk;
    int nc;
    unsigned flags;
};

template <int D, bool FP8>
cudaError_t launch_split(int nr, unsigned grid, cudaStream_t st, const CUtensorMap& mk,
                         const CUtensorMap& mv, const DecodeParams& dp)
{
    if (nr == 2)
        return launch_pdl(paged_decode_prefix_kernel<D, FP8>, grid, Geom<D, FP8>::WARPS * 32,
                          Geom<D, FP8>::SMEM, st, mk, mv, dp);
    return launch_pdl(paged_decode_split_kernel<D, FP8>, grid, Geom<D, FP8>::WARPS * 32, Geom<D, FP8>::SMEM,
                      st, mk, mv, dp);
}

// Validate, build the tensor maps and launch the split and merge kernels.
int decode_launch(void* out, int out_dtype, const void* q, const void* k_cache,
                  const void* v_cache, int kv_dtype, float k_scale, float v_scale, int num_blocks,
                  const int32_t* block_tables, int max_blocks_per_seq,
                  const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                  int head_dim, float scale, void* workspace, size_t workspace_bytes,
                  void* stream, const AppendArgs* app, const PrefixArgs* pre, void* ev_begin,
                  void* ev_split, void* ev_end)
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
    const int nc = pre ? pre->nc : 0;
    if (nc < 0 || nc > num_seqs / 2) return KV_ERR_INVALID_ARG;
    if (nc > 0 && (!pre->chunk || !pre->seq_chunk)) return KV_ERR_INVALID_ARG;
    const bool fp8 = kv_dtype == KV_DTYPE_FP8_E4M3;
    if (fp8 && !(k_scale > 0.f && v_scale > 0.f && std::isfinite(k_scale) && std::isfinite(v_scale)))
        return KV_ERR_INVALID_ARG;
    HeadSplit hs0;
    if (int rc = head_split(num_q_heads, num_kv_heads, hs0)) return rc;
    // flat work indices and tensor-map rows must fit in int32
    if (((long long)num_seqs + nc) * max_blocks_per_seq * hs0.Hkv_v >= INT_MAX ||
        (long long)num_blocks * num_kv_heads >= INT_MAX ||
        (long long)max_blocks_per_seq * kBlock >= INT_MAX)
        return KV_ERR_UNSUPPORTED;

    // one launch: the 16-row kernel (prefix chunks, then sequences; or
    // groups of 9-16 rows) or the plain one; with chunks each phase has its
    // own partial slots
    LaunchPlan lp;
    if (int rc = plan_launch(num_seqs, nc, num_q_heads, num_kv_heads, head_dim, fp8, lp))
        return rc;
    const int nr = lp.nr, grid = lp.grid, warps_total = lp.warps_total;
    const int slot_warps = lp.slot_warps;
    const int Hkv_v = lp.hs.Hkv_v;
    const WsLayout ws = lp.ws;
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
    dp.pair_meta = reinterpret_cast<int4*>(wsb + ws.meta);
    dp.k_new = app ? static_cast<const uint16_t*>(app->k_new) : nullptr;
    dp.v_new = app ? static_cast<const uint16_t*>(app->v_new) : nullptr;
    dp.k_cache = app ? static_cast<uint8_t*>(app->k_cache) : nullptr;
    dp.v_cache = app ? static_cast<uint8_t*>(app->v_cache) : nullptr;
    dp.B = num_seqs;
    dp.Hq = num_q_heads;
    dp.Hkv = Hkv_v;
    dp.G = lp.hs.G_v;
    dp.hshift = lp.hs.hshift;
    dp.Hkv_p = num_kv_heads;
    dp.team_slots = (num_seqs + nc) * num_kv_heads + (warps_total >> lp.hs.hshift);
    dp.max_blocks = max_blocks_per_seq;
    dp.num_blocks = num_blocks;
    dp.warps_total = warps_total;
    dp.min_q1 = std::min(kMinBlocksPerWarp,
                         std::max(2, (max_blocks_per_seq + kMergeDirect - 1) / kMergeDirect));
    dp.sl2 = scale * 1.4426950408889634f * (fp8 ? k_scale : 1.f);
    dp.v_scale = fp8 ? v_scale : 1.f;
    dp.k_qscale = k_scale;
    dp.v_qscale = v_scale;
    dp.out_f32 = out_dtype == KV_DTYPE_F32;
    dp.chunk = nc > 0 ? pre->chunk : nullptr;
    dp.seq_chunk = nc > 0 ? pre->seq_chunk : nullptr;
    dp.nc = nc;
    dp.prow = nr == 2 ? KV_PREFIX_MAX_ROWS : dp.G;
    dp.slot_base = nc > 0 ? warps_total : 0;
    dp.early = pre && (pre->flags & KV_DECODE_EARLY_INPUTS) ? 1 : 0;
    dp.test_stall = g_test_stall.load(std::memory_order_relaxed);

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (ev_begin && cudaEventRecord(static_cast<cudaEvent_t>(ev_begin), st) != cudaSuccess)
        return KV_ERR_CUDA;
    cudaError_t err;
    if (lp.wide) {
        WideParams wp;
        wp.q = dp.q;
        wp.out = out;
        wp.bt = block_tables;
        wp.ctx = context_lens;
        wp.part_o = dp.part_o;
        wp.part_ml = dp.part_ml;
        wp.pair_meta = dp.pair_meta;
        wp.k_new = dp.k_new;
        wp.v_new = dp.v_new;
        wp.k_cache = dp.k_cache;
        wp.v_cache = dp.v_cache;
        wp.B = num_seqs;
        wp.Hq = num_q_heads;
        wp.Hkv_p = num_kv_heads;
        wp.G = num_q_heads / num_kv_heads;
        wp.Gv = lp.hs.G_v;
        wp.hshift = lp.hs.hshift;
        wp.max_blocks = max_blocks_per_seq;
        wp.num_blocks = num_blocks;
        wp.nctas = grid;
        wp.min_q = dp.min_q1;
        wp.team_slots = num_seqs * num_kv_heads + grid;
        wp.sl2 = dp.sl2;
        wp.out_f32 = dp.out_f32;
        wp.early = dp.early;
        wp.test_stall = dp.test_stall;
        err = wide_launch(mk, mv, wp, st);
    } else if (head_dim == 128) {
        err = fp8 ? launch_split<128, true>(nr, grid, st, mk, mv, dp)
                  : launch_split<128, false>(nr, grid, st, mk, mv, dp);
    } else {
        err = fp8 ? launch_split<64, true>(nr, grid, st, mk, mv, dp)
                  : launch_split<64, false>(nr, grid, st, mk, mv, dp);
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
    mp.chunk = dp.chunk;
    mp.seq_chunk = dp.seq_chunk;
    mp.nc = nc;
    mp.prow = dp.prow;
    mp.B = num_seqs;
    mp.Hq = num_q_heads;
    mp.Hkv = Hkv_v;
    mp.G = dp.G;
    mp.max_blocks = max_blocks_per_seq;
    mp.nslots = (num_seqs + nc) * Hkv_v + slot_warps;
    mp.out_f32 = dp.out_f32;
    mp.early = dp.early;
    // one CTA per (sequence, KV head) while that fills the GPU; fewer pairs
    // than SMs (long contexts at small batch: many partials per pair) take
    // one CTA per query row, as long as those are at most two per SM (more,
    // small CTAs cost more to schedule than the split of each pair's
    // partials saves: measured on 64-row MQA, 32 x 8193)
    const int msms = num_sms_current();
    const int mpairs = num_seqs * Hkv_v;
    if (mpairs >= msms || mpairs * dp.G > 2 * msms) {
        const unsigned mgrid = (unsigned)(num_seqs * Hkv_v);
        const unsigned mthreads = (unsigned)merge_threads(dp.G, head_dim);
        err = head_dim == 128
                  ? launch_pdl(paged_decode_merge_kernel<128>, mgrid, mthreads, 0, st, mp)
                  : launch_pdl(paged_decode_merge_kernel<64>, mgrid, mthreads, 0, st, mp);
    } else {
        const unsigned mgrid = (unsigned)(num_seqs * Hkv_v * dp.G);
        const unsigned mthreads = (unsigned)(kMergeRowWarps * 32);
        err = head_dim == 128
                  ? launch_pdl(paged_decode_merge_row_kernel<128>, mgrid, mthreads, 0, st, mp)
                  : launch_pdl(paged_decode_merge_row_kernel<64>, mgrid, mthreads, 0, st, mp);
    }
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
constexpr size_t kStaticWorkspaceBytes = KV_NOALLOC_WORKSPACE_BYTES;     // 16 MiB
static_assert(kStaticWorkspaceBytes == (size_t)16 << 20, "the size the header promises");
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
    LaunchPlan lp;
    if (int rc = plan_launch(num_seqs, 0, num_q_heads, num_kv_heads, head_dim,
                             kv_dtype == KV_DTYPE_FP8_E4M3, lp))
        return rc;
    *bytes = lp.ws.total;
    return KV_OK;
}

extern "C" int paged_decode_prefix_workspace_bytes(int num_seqs, int num_chunks, int num_q_heads,
                                                   int num_kv_heads, int head_dim, int kv_dtype,
                                                   size_t* bytes)
{
    if (!bytes) return KV_ERR_INVALID_ARG;
    *bytes = 0;
    if (int rc = check_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, kv_dtype)) return rc;
    if (num_chunks < 0 || num_chunks > num_seqs / 2) return KV_ERR_INVALID_ARG;
    LaunchPlan lp;
    if (int rc = plan_launch(num_seqs, num_chunks, num_q_heads, num_kv_heads, head_dim,
                             kv_dtype == KV_DTYPE_FP8_E4M3, lp))
        return rc;
    *bytes = lp.ws.total;
    return KV_OK;
}

extern "C" int paged_decode(void* out, int out_dtype, const void* q, const void* k_new,
                            const void* v_new, void* k_cache, void* v_cache, int kv_dtype,
                            float k_scale, float v_scale, int num_blocks,
                            const int32_t* block_tables, int max_blocks_per_seq,
                            const int32_t* context_lens, int num_seqs, int num_q_heads,
                            int num_kv_heads, int head_dim, float scale, const int32_t* chunks,
                            const int32_t* seq_chunk, int num_chunks, unsigned flags,
                            void* workspace, size_t workspace_bytes, void* stream)
{
    if ((k_new == nullptr) != (v_new == nullptr)) return KV_ERR_INVALID_ARG;
    if (flags & ~KV_DECODE_EARLY_INPUTS) return KV_ERR_INVALID_ARG;
    const AppendArgs app = {k_new, v_new, k_cache, v_cache};
    const PrefixArgs pre = {chunks, seq_chunk, num_chunks, flags};
    return decode_launch(out, out_dtype, q, k_cache, v_cache, kv_dtype, k_scale, v_scale,
                         num_blocks, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                         num_q_heads, num_kv_heads, head_dim, scale, workspace, workspace_bytes,
                         stream, k_new ? &app : nullptr, &pre, nullptr, nullptr, nullptr);
}

extern "C" int paged_decode_timed(void* out, int out_dtype, const void* q, const void* k_new,
                                  const void* v_new, void* k_cache, void* v_cache, int kv_dtype,
                                  float k_scale, float v_scale, int num_blocks,
                                  const int32_t* block_tables, int max_blocks_per_seq,
                                  const int32_t* context_lens, int num_seqs, int num_q_heads,
                                  int num_kv_heads, int head_dim, float scale,
                                  const int32_t* chunks, const int32_t* seq_chunk,
                                  int num_chunks, unsigned flags, void* workspace,
                                  size_t workspace_bytes, void* stream, void* ev_begin,
                                  void* ev_split_end, void* ev_end)
{
    if ((k_new == nullptr) != (v_new == nullptr)) return KV_ERR_INVALID_ARG;
    if (flags & ~KV_DECODE_EARLY_INPUTS) return KV_ERR_INVALID_ARG;
    const AppendArgs app = {k_new, v_new, k_cache, v_cache};
    const PrefixArgs pre = {chunks, seq_chunk, num_chunks, flags};
    return decode_launch(out, out_dtype, q, k_cache, v_cache, kv_dtype, k_scale, v_scale,
                         num_blocks, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                         num_q_heads, num_kv_heads, head_dim, scale, workspace, workspace_bytes,
                         stream, k_new ? &app : nullptr, &pre, ev_begin, ev_split_end, ev_end);
}

extern "C" int kv_prefix_plan(const int32_t* block_tables, int max_blocks_per_seq,
                              const int32_t* context_lens, int num_seqs, int num_q_heads,
                              int num_kv_heads, int head_dim, int kv_dtype, int resident_warps,
                              int32_t* chunks, int32_t* seq_chunk, int* num_chunks)
{
    if (!num_chunks) return KV_ERR_INVALID_ARG;
    *num_chunks = 0;
    if (int rc = check_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, kv_dtype)) return rc;
    if (resident_warps <= 0) {
        // the plain split kernel's persistent grid on the current device
        int sms = 0, cps = 0;
        if (int rc = device_info(head_dim, kv_dtype == KV_DTYPE_FP8_E4M3, 1, sms, cps)) return rc;
        resident_warps = sms * cps * warps_per_cta(head_dim, kv_dtype == KV_DTYPE_FP8_E4M3);
    }
    return prefix_plan_host(block_tables, max_blocks_per_seq, context_lens, num_seqs,
                            num_q_heads / num_kv_heads, num_kv_heads, resident_warps, chunks,
                            seq_chunk, num_chunks);
}

extern "C" int kv_test_pipeline_stall(long long cycles)
{
    if (cycles < 0 || cycles > kWaitLimit) return KV_ERR_INVALID_ARG;
    g_test_stall.store(cycles, std::memory_order_relaxed);
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
                         stream, nullptr, nullptr, ev_begin, ev_split_end, ev_end);
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
                         stream, nullptr, nullptr, nullptr, nullptr, nullptr);
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
                         stream, &app, nullptr, nullptr, nullptr, nullptr);
}

extern "C" int kv_get_device_error(int* flags, int64_t* detail)
{
    unsigned f1 = 0, f2 = 0, f3 = 0;
    long long d1 = -1, d2 = -1, d3 = -1;
    if (int rc = append_read_error(&f1, &d1)) return rc;
    if (int rc = decode_read_error(&f2, &d2)) return rc;
    if (int rc = wide_read_error(&f3, &d3)) return rc;
    if (flags) *flags = (int)(f1 | f2 | f3);
    if (detail) *detail = f1 ? d1 : (f2 ? d2 : d3);
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
