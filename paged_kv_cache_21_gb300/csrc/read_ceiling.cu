// kv_read_ceiling: a measurement hook, not part of the decode path.
//
// Streams a device buffer into shared memory with bulk copies and does no
// arithmetic on it, in the same pattern the split-KV decode kernel uses for
// its cache tiles: a persistent grid, 4 warps per CTA, each warp an equal
// contiguous range of 8 KB pieces behind a ring of 3 stages on mbarriers
// (24 KB in flight per warp), copies issued by lane 0 with the L2
// evict-first hint.  Its bandwidth is the read rate the decode kernel could
// reach if its math were free -- a read-only ceiling, beside the copy
// benchmark's read + write figure.
#include <cuda_runtime.h>

#include <mutex>

#include "device_common.cuh"
#include "internal.h"
#include "paged_kv.h"

namespace pkv {

namespace {

constexpr int kRcWarps = 4;
constexpr int kRcStages = 3;
constexpr int kRcPiece = 8192;                 // bytes per bulk copy (one K+V stage at d128 bf16)
constexpr long long kRcWaitLimit = 1LL << 31;  // ~1 s of SM clocks
constexpr int kRcBarOff = kRcWarps * kRcStages * kRcPiece;
constexpr int kRcSmem = kRcBarOff + kRcWarps * kRcStages * 8 + 128;

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// sink[0]: XOR of the first word of every piece (keeps the reads observable);
// sink[1]: set to 1 if a copy never arrived (the warp then stops, after its
// copies in flight have landed or their waits have run out).
__global__ void __launch_bounds__(kRcWarps * 32) read_ceiling_kernel(const uint8_t* src,
                                                                      long long bytes,
                                                                      unsigned* sink)
{
    extern __shared__ uint8_t smem_raw[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t sbase = (smem_u32(smem_raw) + 127u) & ~127u;
    const uint32_t stage0 = sbase + (uint32_t)(warp * kRcStages * kRcPiece);
    const uint32_t bar0 = sbase + (uint32_t)(kRcBarOff + warp * kRcStages * 8);

    const long long pieces = (bytes + kRcPiece - 1) / kRcPiece;
    const long long W = (long long)gridDim.x * kRcWarps;
    const long long w = (long long)blockIdx.x * kRcWarps + warp;
    const long long per = (pieces + W - 1) / W;
    const long long p0 = w * per;
    const long long n = p0 < pieces ? (pieces - p0 < per ? pieces - p0 : per) : 0;
    if (n <= 0) return;

    if (lane == 0) {
        for (int st = 0; st < kRcStages; ++st) mbar_init(bar0 + st * 8, 1);
        fence_mbar_init();
    }
    __syncwarp();
    const uint64_t pol = l2_evict_first_policy();
    auto issue = [&](long long i, int st) {
        if (lane == 0) {
            const long long off = (p0 + i) * kRcPiece;
            const uint32_t sz = (uint32_t)(bytes - off < kRcPiece ? bytes - off : kRcPiece);
            const uint32_t bar = bar0 + st * 8;
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(bar, sz);
            bulk_load(stage0 + (uint32_t)(st * kRcPiece), src + off, sz, bar, pol);
        }
    };
    const int npro = n < kRcStages ? (int)n : kRcStages;
    for (int j = 0; j < npro; ++j) issue(j, j);

    unsigned acc = 0;
    int st = 0;
    uint32_t phase = 0;
    for (long long i = 0; i < n; ++i) {
        bool ok = true;
        if (lane == 0) ok = mbar_wait_bounded(bar0 + st * 8, phase, kRcWaitLimit);
        ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
        if (!ok) {
            if (lane == 0) {
                atomicOr(sink + 1, 1u);
                // the copies of pieces (i, i + stages) are still in flight
                int s2 = st;
                uint32_t ph2 = phase;
                for (long long j = i; j < n && j < i + kRcStages; ++j) {
                    mbar_wait_bounded(bar0 + s2 * 8, ph2, kRcWaitLimit);
                    if (++s2 == kRcStages) { s2 = 0; ph2 ^= 1u; }
                }
            }
            __syncwarp();
            return;
        }
        if (lane == 0) {
            uint32_t v;
            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(stage0 + st * kRcPiece));
            acc ^= v;
        }
        __syncwarp();
        if (i + kRcStages < n) issue(i + kRcStages, st);
        if (++st == kRcStages) { st = 0; phase ^= 1u; }
    }
    if (lane == 0) atomicXor(sink, acc);
}

std::mutex g_rc_mu;
bool g_rc_ready[64] = {};
int g_rc_ctas[64] = {};

}  // namespace

}  // namespace pkv

using namespace pkv;

extern "C" int kv_read_ceiling(const void* buf, size_t bytes, unsigned* sink, void* stream)
{
    if (!buf || !sink || bytes == 0 || bytes % 16 != 0) return KV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(buf) & 15) != 0 || (reinterpret_cast<uintptr_t>(sink) & 3) != 0)
        return KV_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KV_ERR_CUDA;
    int ctas = 0;
    {
        std::lock_guard<std::mutex> lk(g_rc_mu);
        if (!g_rc_ready[dev]) {
            if (cudaFuncSetAttribute(read_ceiling_kernel,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kRcSmem) != cudaSuccess)
                return KV_ERR_CUDA;
            int n = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, read_ceiling_kernel,
                                                              kRcWarps * 32, kRcSmem) !=
                    cudaSuccess ||
                n <= 0)
                return KV_ERR_CUDA;
            g_rc_ctas[dev] = n;
            g_rc_ready[dev] = true;
        }
        ctas = g_rc_ctas[dev];
    }
    const int grid = num_sms_current() * ctas;
    read_ceiling_kernel<<<grid, kRcWarps * 32, kRcSmem, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t*>(buf), (long long)bytes, sink);
    return cudaGetLastError() == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}
