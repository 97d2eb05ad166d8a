// Host-side declarations shared between the translation units of libpagedkv.
#pragma once

#include <cstdint>

namespace pkv {

// Number of SMs of the current device (cached per device), or 1 on error.
int num_sms_current();

// Read and clear the sticky device error word of one translation unit.
int append_read_error(unsigned* flags, long long* detail);
int decode_read_error(unsigned* flags, long long* detail);

// The decision of kv_prefix_plan for a given number of resident warps of the
// split-KV kernel (host only; allocator.cpp).
int prefix_plan_host(const int32_t* block_tables, int max_blocks_per_seq,
                     const int32_t* context_lens, int num_seqs, int group_size,
                     int num_kv_heads, int resident_warps, int32_t* chunks, int32_t* seq_chunk,
                     int* num_chunks);

}  // namespace pkv
