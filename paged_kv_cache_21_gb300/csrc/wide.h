// The wide-group decode kernel (query groups of 17-128 rows per KV head on
// 5th-generation tensor cores): parameters and host entry points shared by
// the CUDA translation units of libpagedkv.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace pkv {

struct WideParams {
    const uint16_t* q;         // bf16 [B][Hq][128]
    void* out;                 // [B][Hq][128], bf16 or f32
    const int32_t* bt;         // [B][max_blocks]
    const int32_t* ctx;        // [B]
    float* part_o;             // partial outputs [slots][16][128]
    float2* part_ml;           // their (max in log2 units, sum) [slots][16]
    int4* pair_meta;           // [B * Hkv_p << hshift]: (first slot, partials, -1, 0)
    const uint16_t* k_new;     // bf16 [B][Hkv_p][128] or null: no append
    const uint16_t* v_new;
    uint8_t* k_cache;          // written by the fused append only
    uint8_t* v_cache;
    int B, Hq, Hkv_p;          // sequences, query heads, (physical) KV heads
    int G;                     // query heads per KV head (17..128)
    int Gv, hshift;            // the merge's sub-groups: 1 << hshift of Gv <= 16 rows
    int max_blocks, num_blocks;
    int nctas;                 // persistent grid
    int min_q;                 // minimum units per CTA
    int team_slots;            // partial slots of one sub-group: B * Hkv_p + nctas
    float sl2;                 // scale * log2(e)
    int out_f32;
    int early;                 // read tables and caches before the dependency wait
    long long test_stall;      // > 0: test hook, see kv_test_pipeline_stall
};

// The CTAs one SM holds of the instantiation a group of G rows uses (cached
// per device).
int wide_setup(int G, int& ctas_per_sm);
// Launch with programmatic stream serialisation; grid = p.nctas.
cudaError_t wide_launch(const CUtensorMap& mk, const CUtensorMap& mv, const WideParams& p,
                        cudaStream_t st);
int wide_read_error(unsigned* flags, long long* detail);

}  // namespace pkv
