// kv_append and kv_copy_blocks: the writes into the paged cache.
//
// The new token's K/V goes to its slot (block * 16 + offset) before the query
// attends ("Transformer attention mask and KV cache inference", section
// "Prefill and decode phases").  With an FP8 cache each element is stored as
// E4M3(x / scale) ("KV cache complete guide", section "(1) FP8
// quantization").  Copy-on-write of a shared block ("KV cache complete
// guide", section "(4) PagedAttention") is a whole-block copy.
//
// Both kernels are pure streaming: one thread moves one 16-byte chunk (8
// bfloat16 in, 16 or 8 bytes out), so every global access is a fully used
// 16-byte vector; the grid is sized in multiples of the SM count.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"
#include "paged_kv.h"

namespace pkv {

__device__ DevErr g_append_err;

template <bool FP8>
__global__ void __launch_bounds__(256) kv_append_kernel(const uint4* __restrict__ k,
                                                        const uint4* __restrict__ v,
                                                        uint8_t* __restrict__ k_cache,
                                                        uint8_t* __restrict__ v_cache,
                                                        const int64_t* __restrict__ slots,
                                                        int num_tokens, int chunks_per_token,
                                                        int chunks_per_head, long long num_slots,
                                                        float k_scale, float v_scale)
{
    // chunk index space: [tensor (K, V)][token][head][chunk of 8 elements]
    const long long per_tensor = (long long)num_tokens * chunks_per_token;
    const long long total = 2 * per_tensor;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const bool is_v = idx >= per_tensor;
        const long long r = is_v ? idx - per_tensor : idx;
        const int tok = (int)(r / chunks_per_token);
        const int rem = (int)(r - (long long)tok * chunks_per_token);
        const int head = rem / chunks_per_head;
        const int c = rem - head * chunks_per_head;
        const long long slot = __ldg(slots + tok);
        if (slot < 0) continue;                           // padding token
        if (slot >= num_slots) {
            raise_flag(&g_append_err, KV_DEVERR_SLOT_OUT_OF_RANGE, slot);
            continue;
        }
        const int num_heads = chunks_per_token / chunks_per_head;
        const long long blk = slot >> 4, off = slot & 15;
        // element offset of (blk, head, off, 8c) in [NB][Hkv][16][D]
        const long long D = (long long)chunks_per_head * 8;
        const long long dst = ((blk * num_heads + head) * kBlock + off) * D + 8LL * c;
        const uint4 x = __ldg((is_v ? v : k) + r);
        uint8_t* cache = is_v ? v_cache : k_cache;
        if (!FP8) {
            *reinterpret_cast<uint4*>(cache + dst * 2) = x;
        } else {
            *reinterpret_cast<uint2*>(cache + dst) = quantize8_e4m3(x, is_v ? v_scale : k_scale);
        }
    }
}

// Copy whole (block, all heads) tiles: chunk space [tensor][pair][16-byte chunk].
__global__ void __launch_bounds__(256) kv_copy_blocks_kernel(uint4* __restrict__ k_cache,
                                                             uint4* __restrict__ v_cache,
                                                             const int32_t* __restrict__ src,
                                                             const int32_t* __restrict__ dst,
                                                             int n, int chunks_per_block,
                                                             int num_blocks)
{
    const long long per_tensor = (long long)n * chunks_per_block;
    const long long total = 2 * per_tensor;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const bool is_v = idx >= per_tensor;
        const long long r = is_v ? idx - per_tensor : idx;
        const int i = (int)(r / chunks_per_block);
        const int c = (int)(r - (long long)i * chunks_per_block);
        const int s = __ldg(src + i), d = __ldg(dst + i);
        if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
            raise_flag(&g_append_err, KV_DEVERR_BLOCK_OUT_OF_RANGE, (s < 0 || s >= num_blocks) ? s : d);
            continue;
        }
        uint4* cache = is_v ? v_cache : k_cache;
        cache[(long long)d * chunks_per_block + c] = cache[(long long)s * chunks_per_block + c];
    }
}

int append_read_error(unsigned* flags, long long* detail)
{
    DevErr e;
    if (cudaMemcpyFromSymbol(&e, g_append_err, sizeof e) != cudaSuccess) return KV_ERR_CUDA;
    DevErr z = {0u, -1LL};
    if (cudaMemcpyToSymbol(g_append_err, &z, sizeof z) != cudaSuccess) return KV_ERR_CUDA;
    *flags = e.flags;
    *detail = e.flags ? e.detail : -1;
    return KV_OK;
}

}  // namespace pkv

using namespace pkv;

extern "C" int kv_append(const void* k, const void* v, void* k_cache, void* v_cache,
                         const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                         int head_dim, int num_blocks, int kv_dtype, float k_scale, float v_scale,
                         void* stream)
{
    if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks <= 0) return KV_ERR_INVALID_ARG;
    if (head_dim <= 0 || head_dim % 8 != 0) return KV_ERR_UNSUPPORTED;
    if (kv_dtype != KV_DTYPE_BF16 && kv_dtype != KV_DTYPE_FP8_E4M3) return KV_ERR_UNSUPPORTED;
    if (num_tokens == 0) return KV_OK;
    if (!k || !v || !k_cache || !v_cache || !slot_mapping) return KV_ERR_INVALID_ARG;
    const uintptr_t align_or = (uintptr_t)k | (uintptr_t)v | (uintptr_t)k_cache |
                               (uintptr_t)v_cache;
    if (align_or & 15) return KV_ERR_INVALID_ARG;
    if (kv_dtype == KV_DTYPE_FP8_E4M3 &&
        !(k_scale > 0.f && v_scale > 0.f && k_scale < 3.0e38f && v_scale < 3.0e38f))
        return KV_ERR_INVALID_ARG;
    const int chunks_per_head = head_dim / 8;
    const int chunks_per_token = chunks_per_head * num_kv_heads;
    const long long total = 2LL * num_tokens * chunks_per_token;
    const int threads = 256;
    long long blocks = (total + threads - 1) / threads;
    const long long cap = (long long)num_sms_current() * 8;
    if (blocks > cap) blocks = cap;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const long long num_slots = (long long)num_blocks * kBlock;
    if (kv_dtype == KV_DTYPE_BF16)
        kv_append_kernel<false><<<(unsigned)blocks, threads, 0, st>>>(
            (const uint4*)k, (const uint4*)v, (uint8_t*)k_cache, (uint8_t*)v_cache, slot_mapping,
            num_tokens, chunks_per_token, chunks_per_head, num_slots, k_scale, v_scale);
    else
        kv_append_kernel<true><<<(unsigned)blocks, threads, 0, st>>>(
            (const uint4*)k, (const uint4*)v, (uint8_t*)k_cache, (uint8_t*)v_cache, slot_mapping,
            num_tokens, chunks_per_token, chunks_per_head, num_slots, k_scale, v_scale);
    return cudaGetLastError() == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

extern "C" int kv_copy_blocks(void* k_cache, void* v_cache, const int32_t* src,
                              const int32_t* dst, int n, int num_kv_heads, int head_dim,
                              int num_blocks, int kv_dtype, void* stream)
{
    if (n < 0 || num_kv_heads <= 0 || num_blocks <= 0 || head_dim <= 0) return KV_ERR_INVALID_ARG;
    if (kv_dtype != KV_DTYPE_BF16 && kv_dtype != KV_DTYPE_FP8_E4M3) return KV_ERR_UNSUPPORTED;
    if (n == 0) return KV_OK;
    if (!k_cache || !v_cache || !src || !dst) return KV_ERR_INVALID_ARG;
    if (((uintptr_t)k_cache | (uintptr_t)v_cache) & 15) return KV_ERR_INVALID_ARG;
    const long long block_bytes =
        (long long)num_kv_heads * kBlock * head_dim * (kv_dtype == KV_DTYPE_BF16 ? 2 : 1);
    if (block_bytes % 16) return KV_ERR_UNSUPPORTED;
    const int chunks_per_block = (int)(block_bytes / 16);
    const long long total = 2LL * n * chunks_per_block;
    const int threads = 256;
    long long blocks = (total + threads - 1) / threads;
    const long long cap = (long long)num_sms_current() * 8;
    if (blocks > cap) blocks = cap;
    kv_copy_blocks_kernel<<<(unsigned)blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(
        (uint4*)k_cache, (uint4*)v_cache, src, dst, n, chunks_per_block, num_blocks);
    return cudaGetLastError() == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}
