// Wide-group decode attention: one decode step for query groups of 17-128
// rows per KV head (MQA on many-head models), bf16 cache, head_dim 128, on
// the 5th-generation tensor cores of sm_103a.
//
// What is computed is the same as paged_decode.cu: for each sequence s and
// query head h (KV head h / G),
//     out[s][h] = softmax_j(scale * q[s][h] . K_j) V_j,   j < context_lens[s]
// ("KV Cache" (heepie.pages.dev), section "Self-Attention"; the length mask of
// "Transformer attention mask and KV cache inference", section "Padding mask
// and batch length"), keys reached through the block table ("KV Cache, Flash
// Attention and inference optimization", section "PagedAttention"), with the
// running (max, sum) softmax of the same lesson's section "Numerical trick".
//
// Why a second kernel: with G query rows per KV head the score and P.V
// contractions are 2 * G * 16 * 128 FLOP per 16-token block and head; at
// G = 64-128 that outgrows warp-level mma.sync (the 16-row kernel then runs
// at a fraction of HBM speed), while a 128-row tcgen05 MMA takes a whole
// group in one instruction.
//
// How:
//  * Persistent grid, two CTAs per SM; each CTA takes an equal contiguous
//    range of the flat (sequence, KV head, block) units.  Warp 4 streams the
//    K and V tiles of its units into a ring of 9 stages (11 when the group has
//    at most 64 rows and Q needs half the buffer) with TMA (the split
//    kernel's tensor maps, 128-byte swizzle; the K tiles of consecutive
//    stages form one contiguous operand) and does the fused append; warp 5
//    allocates tensor memory and issues the score MMAs, warp 6 the P.V MMAs;
//    warps 0-3 own one query row per thread (softmax and output).
//  * Units are consumed in chunks of up to 3 blocks of one (sequence, head)
//    pair.  S = Q K^T: M = 128 query rows (the group, padded), N = 16 keys
//    per block of the chunk in one MMA per 16-wide k-step, K = 128, f32 in
//    tensor memory.  Each row thread loads its row of S (no shuffles),
//    applies the length mask, keeps a reference maximum that moves only when
//    the chunk maximum exceeds it by more than 2^8 (then the accumulator row
//    is rescaled in tensor memory), and stores P = 2^(x - m) split into bf16
//    high and low parts in tensor memory, over the chunk's S.
//    O += P_hi V + P_lo V (A from tensor memory, V as an MN-major operand
//    straight from the ring), f32 in tensor memory.  The score-MMA warp
//    computes the next chunk's scores while the row threads work on this one.
//  * A pair seen whole by one CTA is written normalised; otherwise the CTA
//    stores an unnormalised partial with its (max, sum) per row in the layout
//    of the split kernel's sub-groups of <= 16 rows, and the common merge
//    kernel combines them.
//  * Every wait is bounded; a time-out sets KV_DEVERR_PIPELINE_TIMEOUT and
//    ends every role of the CTA, which still waits for its copies and MMAs in
//    flight before freeing tensor memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "device_common.cuh"
#include "internal.h"
#include "paged_kv.h"
#include "umma.cuh"
#include "wide.h"

namespace pkv {

__device__ DevErr g_wide_err;

namespace {

constexpr int D = 128;
constexpr int kRows = 128;                      // M of every MMA
constexpr int kChunk = 3;                       // blocks per chunk
constexpr int kKeys = kChunk * kBlock;          // keys per chunk (S columns)
constexpr int kBox = kBlock * 128;              // one box: 16 rows x 128 bytes
constexpr uint32_t kTmemCols = 256;
// tensor memory: buffer b at columns 64b holds S of a chunk (48 keys, f32),
// then, in place, its P (bf16 pairs: the high parts from column 64b, the low
// parts from 64b + 32); O at columns 128-255.  Three blocks per chunk rather
// than four: the chunks in the score/softmax/P.V chain hold six ring stages
// instead of eight, so three more blocks are in flight (measured: 64 rows
// 51.1 -> 47.9 us, 128 rows 62.9 -> 57.9 us at 32 x 8193; two blocks per
// chunk: 53.2 and 61.6).
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 128;
constexpr int kThreads = 224;                   // 7 warps
constexpr long long kWaitLimit = 1LL << 31;    // ~1 s of SM clocks
constexpr uint32_t kIdescPV = umma::idesc_bf16_f32(kRows, D, false, true);
static_assert(kKeys == 48, "P stores: one 32-key half, then a 16-key group");

// Shared-memory layout for a Q buffer of QR rows (the group's rows, 64 or
// 128; the 128-row MMAs read rows past QR from the memory that follows, and
// the rows of S they give are never read) and the ring that fills the rest of
// half an SM: the Q rows a group of up to 64 rows leaves free buy two stages.
template <int QR>
struct Layout {
    static constexpr int kRegion = QR * 128;           // QR rows x 128 bytes
    static constexpr int kStages = QR <= 64 ? 11 : 9;  // ring stages (one block's K and V)
    static constexpr int kRingRegion = kStages * kBox; // one box of every stage, contiguous
    static constexpr int kQOff = 0;                    // Q: 2 regions (d 0-63, 64-127)
    static constexpr int kKOff = kQOff + 2 * kRegion;  // K: box 0 of all stages, then box 1
    static constexpr int kVOff = kKOff + 2 * kRingRegion;  // V: likewise
    static constexpr int kBarOff = kVOff + 2 * kRingRegion;
    // barriers
    static constexpr int B_FULL = 0;                   // + stage: the tiles have landed
    static constexpr int B_EMPTY = kStages;            // + stage: the MMAs reading them are done
    static constexpr int B_PATCH = 2 * kStages;        // + stage: the copy warp has edited the tiles
    static constexpr int B_QFULL = 3 * kStages;        // Q of the next segment is in place
    static constexpr int B_INFO = B_QFULL + 1;         // + entry (4): the chunk description is written
    static constexpr int B_INFOFREE = B_INFO + 4;      // + entry (4): the P.V warp has read it
    static constexpr int B_SFULL = B_INFOFREE + 4;     // + buffer (2): S computed
    static constexpr int B_PFULL = B_SFULL + 2;        // + buffer (2): P written
    static constexpr int B_PVDONE = B_PFULL + 2;       // + buffer (2): the P.V MMAs reading that P are done
    static constexpr int B_OFULL = B_PVDONE + 2;       // the segment's accumulator is complete
    static constexpr int B_OFREE = B_OFULL + 1;        // the row threads have read it
    static constexpr int B_FINAL_S = B_OFREE + 1;      // every score MMA of the CTA is done
    static constexpr int B_FINAL_PV = B_FINAL_S + 1;   // every P.V MMA of the CTA is done
    static constexpr int B_STALL = B_FINAL_PV + 1;     // nothing arrives here (the time-out test hook)
    static constexpr int kNumBars = B_STALL + 1;
    static constexpr int kMetaOff = kBarOff + (kNumBars * 8 + 15) / 16 * 16;
    static constexpr int kInfoOff = kMetaOff + kStages * 16;   // 4 entries x 2 int4
    static constexpr int kMiscOff = kInfoOff + 4 * 32;
    static constexpr int kSmem = kMiscOff + 64 + 1024;
    static_assert(kSmem <= 232448 / 2 - 1024, "two CTAs per SM");
    static_assert(kRegion % 1024 == 0 && kRingRegion % 1024 == 0 && kKOff % 1024 == 0,
                  "swizzled operands need 1024-byte aligned atoms");
};

// misc words: [0] tensor-memory base, [1] abort, [2] range start, [3] units,
// [4] units per CTA, [5..7] first unit's (sequence, head, block)
enum Misc { M_TMEM = 0, M_ABORT, M_B0, M_CNT, M_Q, M_S0, M_H0, M_J0 };

// Byte offset of 16-byte chunk c (8 elements) of row r of a stage's tile
// inside its ring (box c / 8 in the second region), as the bulk copy lays
// it out with the 128-byte swizzle (16-byte chunk index XOR row % 8).
template <int RING>
__device__ __forceinline__ uint32_t ring_off(int st, int r, int c)
{
    const uint32_t a = (uint32_t)(r * 128 + (c & 7) * 16);
    return (uint32_t)((c >> 3) * RING + st * kBox) + (a ^ (((a >> 7) & 7u) << 4));
}

// Row r, 16-byte chunk c of a [128 rows x 128 B] region (128-byte swizzle).
__device__ __forceinline__ uint32_t region_off(int r, int c)
{
    return (uint32_t)(r * 128) + (uint32_t)(((c ^ (r & 7)) & 7) * 16);
}

__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Bounded wait that also gives up when another role of the CTA has given up.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* misc)
{
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (misc[M_ABORT]) return false;
        if (clock64() - t0 > kWaitLimit) {
            misc[M_ABORT] = 1;
            raise_flag(&g_wide_err, KV_DEVERR_PIPELINE_TIMEOUT, blockIdx.x);
            return false;
        }
    }
}

__device__ __forceinline__ long long warp_sum_ll(long long v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

__device__ __forceinline__ int seq_blocks_w(const WideParams& p, int s, int& L)
{
    int x = __ldg(p.ctx + s);
    const int cap = p.max_blocks * kBlock;
    if (x < 0 || x > cap) x = x < 0 ? 0 : cap;
    L = x;
    return (x + kBlock - 1) / kBlock;
}

// One unit of a window: lane k of the copy warp holds unit wb + k.
struct WUnit {
    int id, s, h, j, L;
};

// Walk from (s, h, j) forward by `k` units over sequences with blocks.
__device__ __forceinline__ bool advance(const WideParams& p, int& s, int& h, int& j, int& nb,
                                        int& L, int k)
{
    j += k;
    while (j >= nb) {
        j -= nb;
        if (++h == p.Hkv_p) {
            h = 0;
            do {
                if (++s >= p.B) return false;
                nb = seq_blocks_w(p, s, L);
            } while (nb == 0);
        }
    }
    return true;
}

__device__ __forceinline__ void fill_window(const WideParams& p, WUnit& u, int s, int h, int j,
                                            int pos0, int cnt, int lane)
{
    u.id = -1; u.s = 0; u.h = 0; u.j = 0; u.L = 0;
    if (pos0 + lane >= cnt) return;
    int L;
    int nb = seq_blocks_w(p, s, L);
    if (!advance(p, s, h, j, nb, L, lane)) return;
    u.id = __ldg(p.bt + (size_t)s * p.max_blocks + j);
    u.s = s; u.h = h; u.j = j; u.L = L;
}

// The description of a chunk the MMA warp hands to the row threads:
// a = (first unit, blocks, pair, first block), b = (context length of the
// pair, mask of fetched blocks, start | end << 1, segment)
struct ChunkInfo {
    int4 a, b;
};

// ------------------------------------------------------------------ kernel

template <int QR>
__global__ void __launch_bounds__(kThreads, 2)
paged_decode_wide_kernel(const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const WideParams p)
{
    using Ly = Layout<QR>;
    constexpr int kStages = Ly::kStages, kRegion = Ly::kRegion, kRingRegion = Ly::kRingRegion;
    constexpr int kQOff = Ly::kQOff, kKOff = Ly::kKOff, kVOff = Ly::kVOff, kBarOff = Ly::kBarOff;
    constexpr int kMetaOff = Ly::kMetaOff, kInfoOff = Ly::kInfoOff, kMiscOff = Ly::kMiscOff;
    constexpr int B_FULL = Ly::B_FULL, B_EMPTY = Ly::B_EMPTY, B_PATCH = Ly::B_PATCH;
    constexpr int B_QFULL = Ly::B_QFULL, B_INFO = Ly::B_INFO, B_INFOFREE = Ly::B_INFOFREE;
    constexpr int B_SFULL = Ly::B_SFULL, B_PFULL = Ly::B_PFULL, B_PVDONE = Ly::B_PVDONE;
    constexpr int B_OFULL = Ly::B_OFULL, B_OFREE = Ly::B_OFREE, B_FINAL_S = Ly::B_FINAL_S;
    constexpr int B_FINAL_PV = Ly::B_FINAL_PV, B_STALL = Ly::B_STALL;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t sraw = smem_u32(smem_raw);
    const uint32_t sb = (sraw + 1023u) & ~1023u;
    uint8_t* gb = smem_raw + (sb - sraw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int* misc = reinterpret_cast<volatile int*>(gb + kMiscOff);
    int4* meta = reinterpret_cast<int4*>(gb + kMetaOff);
    ChunkInfo* info = reinterpret_cast<ChunkInfo*>(gb + kInfoOff);
    auto bar = [&](int i) -> uint32_t { return sb + (uint32_t)(kBarOff + 8 * i); };
    const int nact = (p.G + 31) / 32;          // row warps with rows of the group

    if (tid == 0) {
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    pdl_launch_dependents();
    if (!p.early) pdl_wait();

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(B_FULL + s), 1);
            mbar_init(bar(B_EMPTY + s), 1);
            mbar_init(bar(B_PATCH + s), 1);
        }
        mbar_init(bar(B_QFULL), nact);
        for (int e = 0; e < 4; ++e) {
            mbar_init(bar(B_INFO + e), 1);
            mbar_init(bar(B_INFOFREE + e), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(B_SFULL + b), 1);
            mbar_init(bar(B_PFULL + b), nact);
            mbar_init(bar(B_PVDONE + b), 1);
        }
        mbar_init(bar(B_OFULL), 1);
        mbar_init(bar(B_OFREE), nact);
        mbar_init(bar(B_FINAL_S), 1);
        mbar_init(bar(B_FINAL_PV), 1);
        mbar_init(bar(B_STALL), 1);
        misc[M_ABORT] = 0;
        fence_mbar_init();
    }
    if (warp == 5) {
        umma::tmem_alloc(sb + kMiscOff + 4 * M_TMEM, kTmemCols);
        umma::tmem_relinquish();
    }
    if (warp == 4) {
        // this CTA's range of the flat (sequence, head, block) units
        long long total = 0;
        for (int base = 0; base < p.B; base += 32) {
            int L, nb = 0;
            if (base + lane < p.B) nb = seq_blocks_w(p, base + lane, L);
            total += warp_sum_ll(nb);
        }
        total *= p.Hkv_p;
        long long q = (total + p.nctas - 1) / p.nctas;
        if (q < p.min_q) q = p.min_q;
        const long long b0 = (long long)blockIdx.x * q;
        long long cnt = total - b0;
        if (cnt > q) cnt = q;
        if (cnt < 0) cnt = 0;
        int s0 = 0, h0 = 0, j0 = 0;
        if (cnt > 0) {
            long long excl = 0;
            bool found = false;
            for (int base = 0; base < p.B && !found; base += 32) {
                int L, nb = 0;
                if (base + lane < p.B) nb = seq_blocks_w(p, base + lane, L);
                const long long v = (long long)nb * p.Hkv_p;
                long long inc = v;
                for (int o = 1; o < 32; o <<= 1) {
                    const long long t = __shfl_up_sync(kFull, inc, o);
                    if (lane >= o) inc += t;
                }
                inc += excl;
                const unsigned m = __ballot_sync(kFull, inc > b0);
                if (m) {
                    const int src = __ffs(m) - 1;
                    const long long ex = __shfl_sync(kFull, inc - v, src);
                    const int nbs = __shfl_sync(kFull, nb, src);
                    s0 = base + src;
                    const long long off = b0 - ex;
                    h0 = (int)(off / nbs);
                    j0 = (int)(off - (long long)h0 * nbs);
                    found = true;
                }
                excl = __shfl_sync(kFull, inc, 31);
            }
            if (!found) cnt = 0;
        }
        if (lane == 0) {
            misc[M_B0] = (int)b0;
            misc[M_CNT] = (int)cnt;
            misc[M_Q] = (int)q;
            misc[M_S0] = s0;
            misc[M_H0] = h0;
            misc[M_J0] = j0;
        }
    }
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = (uint32_t)misc[M_TMEM];
    const int b0 = misc[M_B0], cnt = misc[M_CNT], qper = misc[M_Q];
    const bool append = p.k_new != nullptr;

    if (cnt > 0 && warp == 4) {
        // ------------------------------------------------------------- copies
        WUnit cur, nxt;
        int wb = 0;
        const int s0 = misc[M_S0], h0 = misc[M_H0], j0 = misc[M_J0];
        fill_window(p, cur, s0, h0, j0, 0, cnt, lane);
        auto refill = [&](int pos0) {
            int s = __shfl_sync(kFull, cur.s, 31), h = __shfl_sync(kFull, cur.h, 31);
            int j = __shfl_sync(kFull, cur.j, 31);
            int L, nb = seq_blocks_w(p, s, L);
            if (!advance(p, s, h, j, nb, L, 1)) { nxt.id = -1; return; }
            fill_window(p, nxt, s, h, j, pos0, cnt, lane);
        };
        if (cnt > 32) refill(32);
        const uint64_t pol = l2_evict_first_policy();
        bool waited = !p.early;
        int issued = 0;
        for (int i = 0; i < cnt; ++i) {
            if (i == wb + 32) {
                cur = nxt;
                wb += 32;
                if (wb + 32 < cnt) refill(wb + 32);
            }
            const int src = i - wb;
            const int id = __shfl_sync(kFull, cur.id, src);
            const int s = __shfl_sync(kFull, cur.s, src);
            const int h = __shfl_sync(kFull, cur.h, src);
            const int j = __shfl_sync(kFull, cur.j, src);
            const int L = __shfl_sync(kFull, cur.L, src);
            const int st = i % kStages, round = i / kStages;
            bool ok = true;
            if (round > 0 && lane == 0)
                ok = wait_bar(bar(B_EMPTY + st), (uint32_t)((round - 1) & 1), misc);
            if (!__shfl_sync(kFull, ok ? 1 : 0, 0)) break;
            const bool valid = id >= 0 && id < p.num_blocks;
            const int nb = (L + kBlock - 1) / kBlock;
            const int nvalid = L - j * kBlock;
            const bool fix = !valid || (j == nb - 1 && (append || nvalid < kBlock));
            const uint32_t kst = sb + kKOff, vst = sb + kVOff;
            const uint32_t fb = bar(B_FULL + st);
            if (lane == 0) {
                meta[st] = make_int4(s * p.Hkv_p + h, j, L, (valid ? 1 : 0) | (fix ? 2 : 0));
                if (valid) {
                    mbar_arrive_expect_tx(fb, (uint32_t)(4 * kBox));
                } else {
                    raise_flag(&g_wide_err, KV_DEVERR_BLOCK_OUT_OF_RANGE, id);
                    mbar_arrive(fb);
                }
            }
            __syncwarp();
            // the four boxes of the unit (K and V, d 0-63 and 64-127) are issued
            // by four lanes in one instruction
            if (valid && lane < 4) {
                const int z = id * p.Hkv_p + h;
                const uint32_t dst = (lane < 2 ? kst : vst) + (uint32_t)((lane & 1) * kRingRegion + st * kBox);
                tma_load_3d_hint(dst, lane < 2 ? &tm_k : &tm_v, (lane & 1) * 64, 0, z, fb, pol);
            }
            issued = i + 1;
            if (fix) {
                // the tile must have landed before it is edited
                ok = true;
                if (valid && lane == 0) ok = wait_bar(bar(B_FULL + st), (uint32_t)(round & 1), misc);
                if (!__shfl_sync(kFull, ok ? 1 : 0, 0)) break;
                if (!waited) {
                    pdl_wait();
                    waited = true;
                }
                if (!valid) {
                    // no copy: a zero V tile (the row threads mask every key)
                    for (int c = lane; c < kBlock * 16; c += 32)
                        sts128(vst + ring_off<kRingRegion>(st, c >> 4, c & 15), make_uint4(0, 0, 0, 0));
                } else {
                    if (append && j == nb - 1) {
                        // the step's new token: position L - 1 of its last block
                        const int r = (L - 1) & (kBlock - 1);
                        const bool isv = lane >= 16;
                        const int c = lane & 15;
                        const size_t srco = ((size_t)s * p.Hkv_p + h) * D + 8 * c;
                        const size_t dsto = (((size_t)id * p.Hkv_p + h) * kBlock + r) * D + 8 * c;
                        const uint4 x = __ldg(reinterpret_cast<const uint4*>(
                            (isv ? p.v_new : p.k_new) + srco));
                        *reinterpret_cast<uint4*>((isv ? p.v_cache : p.k_cache) + dsto * 2) = x;
                        sts128((isv ? vst : kst) + ring_off<kRingRegion>(st, r, c), x);
                    }
                    // V rows past the context may hold anything (0 * NaN is NaN)
                    for (int c = lane; c < (kBlock - nvalid) * 16; c += 32)
                        sts128(vst + ring_off<kRingRegion>(st, nvalid + (c >> 4), c & 15),
                               make_uint4(0, 0, 0, 0));
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_PATCH + st));
            }
        }
        // every issued copy lands before the CTA can end
        if (lane == 0) {
            for (int i = issued - kStages < 0 ? 0 : issued - kStages; i < issued; ++i) {
                const int st = i % kStages;
                mbar_wait_bounded(bar(B_FULL + st), (uint32_t)((i / kStages) & 1), kWaitLimit);
            }
        }
        __syncwarp();
    } else if (cnt > 0 && warp == 5) {
        // -------------------------------------------------------------- MMAs
        if (lane == 0) {
            uint32_t patch_phase = 0;            // bit st: parity of stage st's next edit
            // descriptors of the operands' first atoms (start fields advance below)
            const uint64_t qdesc0 = umma::smem_desc_sw128(sb + kQOff, 16, 1024);
            const uint64_t kdesc0 = umma::smem_desc_sw128(sb + kKOff, 16, 1024);
            int seg = -1;
            bool prev_end = true;
            // wait for a chunk's tiles (and edits), describe it to the row threads
            auto plan = [&](int i, int k, ChunkInfo& c) -> bool {
                // test hook: the first wait of the CTA on a barrier that nothing
                // arrives on, for test_stall clocks; every role then stops
                if (k == 0 && p.test_stall > 0 && !mbar_wait_bounded(bar(B_STALL), 0u, p.test_stall)) {
                    misc[M_ABORT] = 1;
                    raise_flag(&g_wide_err, KV_DEVERR_PIPELINE_TIMEOUT, blockIdx.x);
                    return false;
                }
                // entry k & 3 last described chunk k - 4: the P.V warp must be done with it
                if (k >= 4 && !wait_bar(bar(B_INFOFREE + (k & 3)), (uint32_t)(((k - 4) >> 2) & 1), misc))
                    return false;
                const int st = i % kStages;
                if (!wait_bar(bar(B_FULL + st), (uint32_t)((i / kStages) & 1), misc)) return false;
                const int4 m0 = meta[st];
                const int nb = (m0.z + kBlock - 1) / kBlock;
                int n = nb - m0.y;
                if (n > kChunk) n = kChunk;
                if (n > cnt - i) n = cnt - i;
                const bool start = prev_end;
                const bool end = (m0.y + n == nb) || (i + n == cnt);
                if (start) ++seg;
                prev_end = end;
                int vmask = 0;
                for (int u = i; u < i + n; ++u) {
                    const int su = u % kStages;
                    if (u > i &&
                        !wait_bar(bar(B_FULL + su), (uint32_t)((u / kStages) & 1), misc))
                        return false;
                    const int w = meta[su].w;
                    if (w & 1) vmask |= 1 << (u - i);
                    if (w & 2) {
                        if (!wait_bar(bar(B_PATCH + su), (patch_phase >> su) & 1u, misc))
                            return false;
                        patch_phase ^= 1u << su;
                    }
                }
                c.a = make_int4(i, n, m0.x, m0.y);
                c.b = make_int4(m0.z, vmask, (start ? 1 : 0) | (end ? 2 : 0), seg);
                info[k & 3] = c;
                mbar_arrive(bar(B_INFO + (k & 3)));
                return true;
            };
            auto issue_s = [&](const ChunkInfo& c, int k) -> bool {
                const int b = k & 1;
                // buffer b holds P of chunk k - 2 until its P.V products are done
                if (k >= 2 && !wait_bar(bar(B_PVDONE + b), (uint32_t)(((k - 2) >> 1) & 1), misc))
                    return false;
                if ((c.b.z & 1) && !wait_bar(bar(B_QFULL), (uint32_t)(c.b.w & 1), misc))
                    return false;
                umma::fence_after_sync();
                const int i = c.a.x, n = c.a.y;
                const int s0 = i % kStages;
                // the chunk's K rows are contiguous unless its stages wrap
                const int n0 = s0 + n <= kStages ? n : kStages - s0;
                for (int part = 0; part < 2; ++part) {
                    const int np = part == 0 ? n0 : n - n0;
                    if (np <= 0) break;
                    const int sp = part == 0 ? s0 : 0;
                    const uint32_t d = tmem + kColS + (uint32_t)(64 * b + 16 * (part == 0 ? 0 : n0));
                    const uint32_t idesc = umma::idesc_bf16_f32(kRows, 16 * np, false, false);
                    const uint64_t bd0 = kdesc0 + (uint64_t)((sp * kBox) >> 4);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        // the start address field advances by 32 bytes per k-step
                        // inside a 128-byte row, and by a region per 64 elements
                        const uint64_t a = qdesc0 + (uint64_t)(((kk >> 2) * kRegion + (kk & 3) * 32) >> 4);
                        const uint64_t bd = bd0 + (uint64_t)(((kk >> 2) * kRingRegion + (kk & 3) * 32) >> 4);
                        umma::mma_bf16_ss(d, a, bd, idesc, kk > 0);
                    }
                }
                umma::commit(bar(B_SFULL + b));
                return true;
            };
            // the score MMAs of this warp run up to two chunks ahead of the
            // row threads; warp 6 issues the P.V products
            ChunkInfo c;
            int next_i = 0;
            bool ok = true;
            for (int k = 0; ok && next_i < cnt; ++k) {
                ok = plan(next_i, k, c) && issue_s(c, k);
                next_i = c.a.x + c.a.y;
            }
            // every MMA issued by this thread is complete before the CTA ends
            umma::commit(bar(B_FINAL_S));
            mbar_wait_bounded(bar(B_FINAL_S), 0u, kWaitLimit);
        }
        __syncwarp();
    } else if (cnt > 0 && warp == 6) {
        // --------------------------------------------------------- P.V MMAs
        if (lane == 0) {
            const uint64_t vdesc0 = umma::smem_desc_sw128(sb + kVOff, kRingRegion, 1024);
            bool ok = true;
            for (int k = 0; ok; ++k) {
                ok = wait_bar(bar(B_INFO + (k & 3)), (uint32_t)((k >> 2) & 1), misc);
                if (!ok) break;
                const ChunkInfo c = info[k & 3];
                mbar_arrive(bar(B_INFOFREE + (k & 3)));
                const int b = k & 1;
                ok = wait_bar(bar(B_PFULL + b), (uint32_t)((k >> 1) & 1), misc);
                if (!ok) break;
                const bool start = c.b.z & 1;
                if (start && c.b.w > 0) {
                    ok = wait_bar(bar(B_OFREE), (uint32_t)((c.b.w - 1) & 1), misc);
                    if (!ok) break;
                }
                umma::fence_after_sync();
                const int i = c.a.x, n = c.a.y;
                for (int jj = 0; jj < n; ++jj) {
                    const int st = (i + jj) % kStages;
                    const uint64_t bd = vdesc0 + (uint64_t)((st * kBox) >> 4);
                    const uint32_t ph = tmem + kColS + (uint32_t)(64 * b + 8 * jj);
                    umma::mma_bf16_ts(tmem + kColO, ph, bd, kIdescPV, !(start && jj == 0));
                    umma::mma_bf16_ts(tmem + kColO, ph + 32, bd, kIdescPV, true);
                }
                for (int jj = 0; jj < n; ++jj) umma::commit(bar(B_EMPTY + (i + jj) % kStages));
                umma::commit(bar(B_PVDONE + b));
                if (c.b.z & 2) umma::commit(bar(B_OFULL));
                if (i + n >= cnt) break;
            }
            umma::commit(bar(B_FINAL_PV));
            mbar_wait_bounded(bar(B_FINAL_PV), 0u, kWaitLimit);
        }
        __syncwarp();
    } else if (cnt > 0 && warp < nact) {
        // -------------------------------------------------- row threads
        const int r = tid;                       // query row of the group
        const bool live = r < p.G;
        if (p.early) pdl_wait();
        const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
        float m_ref = -INFINITY, l = 0.f;
        int seg_i0 = 0, seg_first = 0, seg_pair = 0, seg_L = 0;
        auto load_q = [&](int pair) {
            if (live) {
                const int s = pair / p.Hkv_p, h = pair - s * p.Hkv_p;
                const uint4* src = reinterpret_cast<const uint4*>(
                    p.q + ((size_t)s * p.Hq + (size_t)h * p.G + r) * D);
                uint4 v[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) v[c] = __ldg(src + c);
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    sts128(sb + kQOff + (uint32_t)((c >> 3) * kRegion) + region_off(r, c & 7), v[c]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_QFULL));
        };
        bool ok = __all_sync(kFull, wait_bar(bar(B_INFO), 0u, misc));
        if (ok) load_q(info[0].a.z);
        for (int k = 0; ok; ++k) {
            ok = __all_sync(kFull, wait_bar(bar(B_INFO + (k & 3)), (uint32_t)((k >> 2) & 1), misc));
            if (!ok) break;
            const ChunkInfo c = info[k & 3];
            const int i = c.a.x, n = c.a.y, blk0 = c.a.w, L = c.b.x, vmask = c.b.y;
            const bool start = c.b.z & 1, end = c.b.z & 2;
            if (start) {
                seg_i0 = i;
                seg_first = blk0;
                seg_pair = c.a.z;
                seg_L = L;
                m_ref = -INFINITY;
                l = 0.f;
            }
            const int b = k & 1;
            ok = __all_sync(kFull, wait_bar(bar(B_SFULL + b), (uint32_t)((k >> 1) & 1), misc));
            if (!ok) break;
            umma::fence_after_sync();
            uint32_t sr[kKeys];
#pragma unroll
            for (int c0 = 0; c0 < kKeys; c0 += 16)
                umma::tmem_ld16(trow + kColS + (uint32_t)(64 * b + c0),
                                *reinterpret_cast<uint32_t(*)[16]>(&sr[c0]));
            umma::tmem_wait_ld();
            const bool more = i + n < cnt;
            // Q is no longer read once this chunk's scores exist: load the
            // next segment's rows now
            if (end && more) {
                ok = __all_sync(kFull, wait_bar(bar(B_INFO + ((k + 1) & 3)),
                                                (uint32_t)(((k + 1) >> 2) & 1), misc));
                if (!ok) break;
                load_q(info[(k + 1) & 3].a.z);
            }
            // raw scores; keys past the context, in blocks that were not
            // fetched, of columns past the chunk and of rows past the group
            // are -inf (the same keys for every row)
            const bool full = n == kChunk && vmask == (1 << kChunk) - 1 &&
                              (blk0 + kChunk) * kBlock <= L && live;
            float* x = reinterpret_cast<float*>(sr);
            // with a negative scale the largest scaled score is the smallest
            // raw one: negate the raw scores and use |scale|
            const float sl2 = fabsf(p.sl2);
            if (p.sl2 < 0.f) {
#pragma unroll
                for (int cc = 0; cc < kKeys; ++cc) x[cc] = -x[cc];
            }
            if (!full) {
#pragma unroll
                for (int cc = 0; cc < kKeys; ++cc) {
                    const int jj = cc >> 4;
                    const bool in = live && jj < n && ((vmask >> jj) & 1) &&
                                    (blk0 + jj) * kBlock + (cc & 15) < L;
                    if (!in) x[cc] = -INFINITY;
                }
            }
            float mr[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int w = kKeys / 8;        // 4 or 8 scores per partial maximum
                float v = x[w * e];
#pragma unroll
                for (int f = 1; f < w; ++f) v = fmaxf(v, x[w * e + f]);
                mr[e] = v;
            }
            const float mraw = fmaxf(fmaxf(fmaxf(mr[0], mr[1]), fmaxf(mr[2], mr[3])),
                                     fmaxf(fmaxf(mr[4], mr[5]), fmaxf(mr[6], mr[7])));
            const float mx = mraw * sl2;        // the max of the scaled scores
            // the reference maximum moves only when the scores outgrow it by
            // more than 2^8; the accumulator row is then rescaled in place
            bool resc = false;
            float alpha = 1.f;
            if (start) {
                m_ref = mx;
            } else if (mx > m_ref + 8.f) {
                alpha = ex2(m_ref - mx);         // 0 while nothing was seen
                m_ref = mx;
                resc = true;
            }
            // P goes over S in buffer b (the S issuer reuses the buffer only
            // after the P.V products of this chunk); a rescale of the
            // accumulator needs those of chunk k - 1
            if (__any_sync(kFull, resc)) {
                ok = __all_sync(kFull, wait_bar(bar(B_PVDONE + ((k - 1) & 1)),
                                                (uint32_t)(((k - 1) >> 1) & 1), misc));
                if (!ok) break;
                umma::fence_after_sync();
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t o[32];
                    umma::tmem_ld32(trow + kColO + (uint32_t)c0, o);
                    umma::tmem_wait_ld();
#pragma unroll
                    for (int cc = 0; cc < 32; ++cc)
                        o[cc] = __float_as_uint(__uint_as_float(o[cc]) * alpha);
                    umma::tmem_st32(trow + kColO + (uint32_t)c0, o);
                }
                l *= alpha;
            }
            // P = 2^(s * scale - m), bf16 high and low parts
            const float nm = m_ref == -INFINITY ? 0.f : -m_ref;
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int half = 0; half < kKeys / 32; ++half) {
                uint32_t hi[16], lo[16];       // keys 32 half .. 32 half + 31
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int cc = 32 * half + 2 * e;
                    float p0 = ex2(fmaf(x[cc], sl2, nm));
                    float p1 = ex2(fmaf(x[cc + 1], sl2, nm));
                    if (!full) {                 // masked keys weigh 0 (also at scale 0)
                        p0 = x[cc] == -INFINITY ? 0.f : p0;
                        p1 = x[cc + 1] == -INFINITY ? 0.f : p1;
                    }
                    ls[e & 3] += p0 + p1;
                    hi[e] = pack_bf16x2(p0, p1);
                    lo[e] = pack_bf16x2(p0 - bf16_lo(hi[e]), p1 - bf16_hi(hi[e]));
                }
                umma::tmem_st16(trow + kColS + (uint32_t)(64 * b + 16 * half), hi);
                umma::tmem_st16(trow + kColS + (uint32_t)(64 * b + 32 + 16 * half), lo);
            }
            if constexpr (kKeys % 32 == 16) {
                // the last 16 keys: 8 columns at a 16-column boundary of each part
                uint32_t hi[8], lo[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int cc = kKeys - 16 + 2 * e;
                    float p0 = ex2(fmaf(x[cc], sl2, nm));
                    float p1 = ex2(fmaf(x[cc + 1], sl2, nm));
                    if (!full) {
                        p0 = x[cc] == -INFINITY ? 0.f : p0;
                        p1 = x[cc + 1] == -INFINITY ? 0.f : p1;
                    }
                    ls[e & 3] += p0 + p1;
                    hi[e] = pack_bf16x2(p0, p1);
                    lo[e] = pack_bf16x2(p0 - bf16_lo(hi[e]), p1 - bf16_hi(hi[e]));
                }
                umma::tmem_st8(trow + kColS + (uint32_t)(64 * b + (kKeys - 16) / 2), hi);
                umma::tmem_st8(trow + kColS + (uint32_t)(64 * b + 32 + (kKeys - 16) / 2), lo);
            }
            l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            umma::tmem_wait_st();
            umma::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_PFULL + b));
            if (end) {
                // the segment's accumulator: output or partial
                ok = __all_sync(kFull, wait_bar(bar(B_OFULL), (uint32_t)(c.b.w & 1), misc));
                if (!ok) break;
                umma::fence_after_sync();
                const int s = seg_pair / p.Hkv_p, h = seg_pair - s * p.Hkv_p;
                const int nbp = (seg_L + kBlock - 1) / kBlock;
                const int last = blk0 + n - 1;
                const bool whole = seg_first == 0 && last == nbp - 1;
                const int sub = live ? r / p.Gv : 0, rr = live ? r - sub * p.Gv : 0;
                const size_t slot = (size_t)sub * p.team_slots + (size_t)seg_pair + blockIdx.x;
                const float inv = l > 0.f ? 1.f / l : 0.f;
                const size_t orow = ((size_t)s * p.Hq + (size_t)h * p.G + (live ? r : 0)) * D;
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t o[32];
                    umma::tmem_ld32(trow + kColO + (uint32_t)c0, o);
                    umma::tmem_wait_ld();
                    if (!live) continue;
                    if (whole) {
                        if (p.out_f32) {
                            float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + orow + c0);
#pragma unroll
                            for (int cc = 0; cc < 32; cc += 4)
                                dst[cc / 4] = make_float4(__uint_as_float(o[cc]) * inv,
                                                          __uint_as_float(o[cc + 1]) * inv,
                                                          __uint_as_float(o[cc + 2]) * inv,
                                                          __uint_as_float(o[cc + 3]) * inv);
                        } else {
                            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.out) + orow + c0);
#pragma unroll
                            for (int cc = 0; cc < 32; cc += 8)
                                dst[cc / 8] = make_uint4(
                                    pack_bf16x2(__uint_as_float(o[cc]) * inv, __uint_as_float(o[cc + 1]) * inv),
                                    pack_bf16x2(__uint_as_float(o[cc + 2]) * inv, __uint_as_float(o[cc + 3]) * inv),
                                    pack_bf16x2(__uint_as_float(o[cc + 4]) * inv, __uint_as_float(o[cc + 5]) * inv),
                                    pack_bf16x2(__uint_as_float(o[cc + 6]) * inv, __uint_as_float(o[cc + 7]) * inv));
                        }
                    } else {
                        float4* dst = reinterpret_cast<float4*>(p.part_o + (slot * 16 + rr) * D + c0);
#pragma unroll
                        for (int cc = 0; cc < 32; cc += 4)
                            dst[cc / 4] = make_float4(__uint_as_float(o[cc]), __uint_as_float(o[cc + 1]),
                                                      __uint_as_float(o[cc + 2]), __uint_as_float(o[cc + 3]));
                    }
                }
                if (live && !whole) p.part_ml[slot * 16 + rr] = make_float2(m_ref, l);
                if (r == 0 && seg_first == 0) {
                    // the CTA holding the pair's first block records where its
                    // partials are: CTAs [this one, the one holding its last unit]
                    const long long flat_first = (long long)b0 + seg_i0;
                    const int c_last = (int)((flat_first + (long long)nbp - 1) / qper);
                    const int npart = c_last - (int)blockIdx.x + 1;
                    const int hv0 = s * (p.Hkv_p << p.hshift) + (h << p.hshift);
                    for (int sb2 = 0; sb2 < (1 << p.hshift); ++sb2)
                        p.pair_meta[hv0 + sb2] = make_int4(
                            (int)((size_t)sb2 * p.team_slots + (size_t)seg_pair + blockIdx.x), npart,
                            -1, 0);
                }
                umma::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_OFREE));
            }
            if (!more) break;
        }
    }

    umma::fence_before_sync();
    __syncthreads();
    if (warp == 5) {
        umma::fence_after_sync();
        umma::tmem_dealloc(tmem, kTmemCols);
    }
}

std::mutex g_wide_mu;
bool g_wide_ready[64][2] = {};
int g_wide_ctas[64][2] = {};

// Q rows of the instantiation a group of G rows uses
inline int qrows_for(int G) { return G <= 64 ? 64 : 128; }

template <int QR>
int wide_setup_variant(int dev, int& n_out)
{
    using Ly = Layout<QR>;
    const auto fn = paged_decode_wide_kernel<QR>;
    // two CTAs per SM need the largest shared-memory carveout
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, Ly::kSmem) !=
            cudaSuccess ||
        cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess)
        return KV_ERR_CUDA;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kThreads, Ly::kSmem) != cudaSuccess)
        return KV_ERR_CUDA;
    // the kernel is sized for two CTAs per SM (shared memory, registers,
    // tensor memory: 2 x 256 of 512 columns); the occupancy query has
    // reported one here while the hardware placed two, so the CTAs per SM
    // are also derived from the function's registers and shared memory
    cudaFuncAttributes fa;
    int smem_sm = 0, smem_rsv = 0, regs_sm = 0;
    if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&smem_rsv, cudaDevAttrReservedSharedMemoryPerBlock, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) !=
            cudaSuccess)
        return KV_ERR_CUDA;
    int by_smem = smem_sm / (Ly::kSmem + (int)fa.sharedSizeBytes + smem_rsv);
    int by_regs = fa.numRegs > 0 ? regs_sm / (fa.numRegs * kThreads) : 1;
    int own = by_smem < by_regs ? by_smem : by_regs;
    if (own > (int)(512 / kTmemCols)) own = 512 / kTmemCols;
    if (own > n) n = own;
    if (n <= 0) return KV_ERR_CUDA;
    n_out = n;
    return KV_OK;
}

}  // namespace

int wide_setup(int G, int& ctas_per_sm)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KV_ERR_CUDA;
    const int v = qrows_for(G) == 64 ? 0 : 1;
    std::lock_guard<std::mutex> lk(g_wide_mu);
    if (!g_wide_ready[dev][v]) {
        int n = 0;
        if (int rc = v == 0 ? wide_setup_variant<64>(dev, n) : wide_setup_variant<128>(dev, n))
            return rc;
        g_wide_ctas[dev][v] = n;
        g_wide_ready[dev][v] = true;
    }
    ctas_per_sm = g_wide_ctas[dev][v];
    return KV_OK;
}

cudaError_t wide_launch(const CUtensorMap& mk, const CUtensorMap& mv, const WideParams& p,
                        cudaStream_t st)
{
    const bool q64 = qrows_for(p.G) == 64;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.nctas);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = q64 ? Layout<64>::kSmem : Layout<128>::kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return q64 ? cudaLaunchKernelEx(&cfg, paged_decode_wide_kernel<64>, mk, mv, p)
               : cudaLaunchKernelEx(&cfg, paged_decode_wide_kernel<128>, mk, mv, p);
}

int wide_read_error(unsigned* flags, long long* detail)
{
    DevErr e;
    if (cudaMemcpyFromSymbol(&e, g_wide_err, sizeof e) != cudaSuccess) return KV_ERR_CUDA;
    DevErr z = {0u, -1LL};
    if (cudaMemcpyToSymbol(g_wide_err, &z, sizeof z) != cudaSuccess) return KV_ERR_CUDA;
    *flags = e.flags;
    *detail = e.flags ? e.detail : -1;
    return KV_OK;
}

}  // namespace pkv
