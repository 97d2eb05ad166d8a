// Host side of the paged KV cache: KV sizing, the block allocator with its free
// list and reference counts, and the per-step slot mapping.
//
// "KV Cache, Flash Attention and inference optimization", section
// "PagedAttention" (16-token blocks, a page table from logical position to
// physical block) and its exercise 3 (a free list; blocks go back to the pool
// when a sequence ends); "KV cache complete guide", section "(4)
// PagedAttention" (requests with a common prefix share physical blocks,
// copy-on-write); "Transformer attention mask and KV cache inference",
// section "Position ID and append contract" (a cache handle owns its length;
// the new token goes at position == current length).
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <map>
#include <new>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "internal.h"
#include "paged_kv.h"

namespace {

struct Seq {
    int64_t len = 0;
    std::vector<int32_t> blocks;
    int32_t slot = -1;         // row in the last kv_step / kv_seq_reorder naming it
    int32_t reorder_src = -1;  // src_index of that row in the last kv_seq_reorder
};

int64_t ceil_blocks(int64_t len) { return (len + KV_BLOCK_SIZE - 1) / KV_BLOCK_SIZE; }

}  // namespace

struct kv_alloc {
    int num_blocks = 0;
    int num_kv_heads = 0;
    int head_dim = 0;
    int kv_dtype = 0;
    std::vector<int32_t> free_list;   // stack; the next block handed out is back()
    std::vector<int32_t> refcount;    // per physical block
    std::unordered_map<int64_t, Seq> seqs;

    int32_t take() {
        int32_t b = free_list.back();
        free_list.pop_back();
        refcount[b] = 1;
        return b;
    }
    void release(int32_t b) {
        if (--refcount[b] == 0) free_list.push_back(b);
    }
};

extern "C" {

int64_t kv_bytes(int layers, int batch, int kv_heads, int64_t seq, int head_dim, int dtype_bytes)
{
    if (layers < 0 || batch < 0 || kv_heads < 0 || seq < 0 || head_dim < 0 || dtype_bytes < 0)
        return -1;
    int64_t r = 2;
    const int64_t f[6] = {layers, batch, kv_heads, seq, head_dim, dtype_bytes};
    for (int64_t x : f)
        if (__builtin_mul_overflow(r, x, &r)) return -1;
    return r;
}

int kv_cache_alloc(kv_alloc_t** out, int num_blocks, int num_kv_heads, int head_dim,
                   int block_size, int kv_dtype)
{
    if (!out) return KV_ERR_INVALID_ARG;
    *out = nullptr;
    if (num_blocks <= 0 || num_kv_heads <= 0 || head_dim <= 0) return KV_ERR_INVALID_ARG;
    if (block_size != KV_BLOCK_SIZE) return KV_ERR_UNSUPPORTED;
    if (kv_dtype != KV_DTYPE_BF16 && kv_dtype != KV_DTYPE_FP8_E4M3) return KV_ERR_UNSUPPORTED;
    kv_alloc* a = new (std::nothrow) kv_alloc;
    if (!a) return KV_ERR_INVALID_ARG;
    a->num_blocks = num_blocks;
    a->num_kv_heads = num_kv_heads;
    a->head_dim = head_dim;
    a->kv_dtype = kv_dtype;
    a->refcount.assign(num_blocks, 0);
    a->free_list.resize(num_blocks);
    // hand out 0, 1, 2, ... first
    for (int i = 0; i < num_blocks; ++i) a->free_list[i] = num_blocks - 1 - i;
    *out = a;
    return KV_OK;
}

void kv_alloc_destroy(kv_alloc_t* a) { delete a; }

int kv_seq_add(kv_alloc_t* a, int64_t seq_id, int64_t len)
{
    if (!a || len < 0) return KV_ERR_INVALID_ARG;
    if (a->seqs.count(seq_id)) return KV_ERR_EXISTS;
    int64_t need = ceil_blocks(len);
    if (need > (int64_t)a->free_list.size()) return KV_ERR_OUT_OF_BLOCKS;
    Seq s;
    s.len = len;
    s.blocks.reserve(need);
    for (int64_t i = 0; i < need; ++i) s.blocks.push_back(a->take());
    a->seqs.emplace(seq_id, std::move(s));
    return KV_OK;
}

int kv_seq_fork(kv_alloc_t* a, int64_t parent, int64_t child, int64_t shared_len)
{
    if (!a || shared_len < 0) return KV_ERR_INVALID_ARG;
    auto it = a->seqs.find(parent);
    if (it == a->seqs.end()) return KV_ERR_NOT_FOUND;
    if (a->seqs.count(child)) return KV_ERR_EXISTS;
    if (shared_len > it->second.len) return KV_ERR_INVALID_ARG;
    Seq s;
    s.len = shared_len;
    int64_t nshare = ceil_blocks(shared_len);
    s.blocks.assign(it->second.blocks.begin(), it->second.blocks.begin() + nshare);
    for (int32_t b : s.blocks) a->refcount[b] += 1;
    a->seqs.emplace(child, std::move(s));
    return KV_OK;
}

int kv_seq_free(kv_alloc_t* a, int64_t seq_id)
{
    if (!a) return KV_ERR_INVALID_ARG;
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return KV_ERR_NOT_FOUND;
    for (int32_t b : it->second.blocks) a->release(b);
    a->seqs.erase(it);
    return KV_OK;
}

int kv_step(kv_alloc_t* a, const int64_t* seq_ids, int n, int64_t* slot_mapping,
            int32_t* block_tables, int max_blocks, int32_t* context_lens, int32_t* cow_src,
            int32_t* cow_dst, int cow_cap, int* n_cow)
{
    if (!a || n < 0 || max_blocks <= 0 || cow_cap < 0) return KV_ERR_INVALID_ARG;
    if (n > 0 && (!seq_ids || !slot_mapping || !block_tables || !context_lens))
        return KV_ERR_INVALID_ARG;
    if (cow_cap > 0 && (!cow_src || !cow_dst)) return KV_ERR_INVALID_ARG;
    if (n_cow) *n_cow = 0;

    // Pass 1: check everything and count the blocks the step needs, simulating
    // the reference-count changes so that two sequences sharing a tail block
    // are handled in order (the first copies, the second then owns it alone).
    std::unordered_set<int64_t> seen;
    std::unordered_map<int32_t, int> ref_delta;
    int64_t need_new = 0, need_cow = 0;
    for (int i = 0; i < n; ++i) {
        auto it = a->seqs.find(seq_ids[i]);
        if (it == a->seqs.end()) return KV_ERR_NOT_FOUND;
        if (!seen.insert(seq_ids[i]).second) return KV_ERR_INVALID_ARG;
        const Seq& s = it->second;
        int64_t pos = s.len;
        if (ceil_blocks(pos + 1) > max_blocks) return KV_ERR_INVALID_ARG;
        if (pos % KV_BLOCK_SIZE == 0) {
            need_new += 1;
        } else {
            int32_t tail = s.blocks[pos / KV_BLOCK_SIZE];
            int rc = a->refcount[tail] + ref_delta[tail];
            if (rc > 1) {
                need_new += 1;
                need_cow += 1;
                ref_delta[tail] -= 1;
            }
        }
    }
    if (need_new > (int64_t)a->free_list.size()) return KV_ERR_OUT_OF_BLOCKS;
    if (need_cow > cow_cap) return KV_ERR_INVALID_ARG;

    // Pass 2: apply.
    int ncow = 0;
    for (int i = 0; i < n; ++i) {
        Seq& s = a->seqs[seq_ids[i]];
        int64_t pos = s.len;
        int64_t bi = pos / KV_BLOCK_SIZE;
        if (pos % KV_BLOCK_SIZE == 0) {
            s.blocks.push_back(a->take());
        } else {
            int32_t tail = s.blocks[bi];
            if (a->refcount[tail] > 1) {
                int32_t fresh = a->take();
                cow_src[ncow] = tail;
                cow_dst[ncow] = fresh;
                ++ncow;
                a->release(tail);
                s.blocks[bi] = fresh;
            }
        }
        slot_mapping[i] = (int64_t)s.blocks[bi] * KV_BLOCK_SIZE + pos % KV_BLOCK_SIZE;
        s.len = pos + 1;
        s.slot = i;
        context_lens[i] = (int32_t)s.len;
        int32_t* row = block_tables + (int64_t)i * max_blocks;
        int nb = (int)s.blocks.size();
        std::memcpy(row, s.blocks.data(), sizeof(int32_t) * nb);
        for (int j = nb; j < max_blocks; ++j) row[j] = -1;
    }
    if (n_cow) *n_cow = ncow;
    return KV_OK;
}

int kv_seq_reorder(kv_alloc_t* a, const int64_t* seq_ids, const int32_t* src_index, int n)
{
    if (!a || n < 0) return KV_ERR_INVALID_ARG;
    if (n == 0) return KV_OK;
    if (!seq_ids || !src_index) return KV_ERR_INVALID_ARG;
    std::unordered_set<int64_t> seen;
    std::vector<Seq*> rows(n);
    for (int i = 0; i < n; ++i) {
        auto it = a->seqs.find(seq_ids[i]);
        if (it == a->seqs.end()) return KV_ERR_NOT_FOUND;
        if (!seen.insert(seq_ids[i]).second) return KV_ERR_INVALID_ARG;
        if (src_index[i] < 0 || src_index[i] >= n) return KV_ERR_INVALID_ARG;
        rows[i] = &it->second;
    }
    // snapshot, then take the new references before dropping the old ones so
    // that a block kept by some row never visits the free list
    std::vector<Seq> old(n);
    for (int i = 0; i < n; ++i) old[i] = *rows[i];
    for (int i = 0; i < n; ++i)
        for (int32_t b : old[src_index[i]].blocks) a->refcount[b] += 1;
    for (int i = 0; i < n; ++i)
        for (int32_t b : old[i].blocks) a->release(b);
    for (int i = 0; i < n; ++i) {
        *rows[i] = old[src_index[i]];
        rows[i]->slot = i;
        rows[i]->reorder_src = src_index[i];
    }
    return KV_OK;
}

int kv_seq_info(kv_alloc_t* a, int64_t seq_id, int64_t* len, int32_t* row, int max_blocks,
                int* nblocks)
{
    if (!a) return KV_ERR_INVALID_ARG;
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return KV_ERR_NOT_FOUND;
    const Seq& s = it->second;
    int nb = (int)s.blocks.size();
    if (row) {
        if (max_blocks < nb) return KV_ERR_INVALID_ARG;
        std::memcpy(row, s.blocks.data(), sizeof(int32_t) * nb);
        for (int j = nb; j < max_blocks; ++j) row[j] = -1;
    }
    if (len) *len = s.len;
    if (nblocks) *nblocks = nb;
    return KV_OK;
}

int kv_alloc_stats(kv_alloc_t* a, int* free_blocks, int* used_blocks, int* num_seqs, int block,
                   int* refcount)
{
    if (!a) return KV_ERR_INVALID_ARG;
    if (free_blocks) *free_blocks = (int)a->free_list.size();
    if (used_blocks) *used_blocks = a->num_blocks - (int)a->free_list.size();
    if (num_seqs) *num_seqs = (int)a->seqs.size();
    if (block >= 0) {
        if (block >= a->num_blocks) return KV_ERR_INVALID_ARG;
        if (refcount) *refcount = a->refcount[block];
    }
    return KV_OK;
}

int kv_alloc_shape(kv_alloc_t* a, int* num_blocks, int* num_kv_heads, int* head_dim,
                   int* kv_dtype)
{
    if (!a) return KV_ERR_INVALID_ARG;
    if (num_blocks) *num_blocks = a->num_blocks;
    if (num_kv_heads) *num_kv_heads = a->num_kv_heads;
    if (head_dim) *head_dim = a->head_dim;
    if (kv_dtype) *kv_dtype = a->kv_dtype;
    return KV_OK;
}

int kv_alloc_trace(kv_alloc_t* a, const int64_t* seq_ids, int n, int64_t* rows, int* count)
{
    if (!a || n < 0) return KV_ERR_INVALID_ARG;
    std::vector<int64_t> ids;
    if (seq_ids) {
        ids.assign(seq_ids, seq_ids + n);
        for (int64_t id : ids)
            if (!a->seqs.count(id)) return KV_ERR_NOT_FOUND;
    } else {
        ids.reserve(a->seqs.size());
        for (const auto& kv : a->seqs) ids.push_back(kv.first);
        std::sort(ids.begin(), ids.end());
        if ((int64_t)ids.size() > n) return KV_ERR_INVALID_ARG;
    }
    if (!ids.empty() && !rows) return KV_ERR_INVALID_ARG;
    const int64_t elt = a->kv_dtype == KV_DTYPE_FP8_E4M3 ? 1 : 2;
    const int64_t block_bytes = 2 * KV_BLOCK_SIZE * (int64_t)a->num_kv_heads * a->head_dim * elt;
    for (size_t r = 0; r < ids.size(); ++r) {
        const Seq& s = a->seqs.find(ids[r])->second;
        int64_t shared = 0;
        for (int32_t b : s.blocks) shared += a->refcount[b] > 1;
        int64_t* row = rows + r * KV_TRACE_FIELDS;
        row[KV_TRACE_SEQ_ID] = ids[r];
        row[KV_TRACE_SLOT] = s.slot;
        row[KV_TRACE_LEN] = s.len;
        row[KV_TRACE_POSITION] = s.len;
        row[KV_TRACE_BLOCKS] = (int64_t)s.blocks.size();
        row[KV_TRACE_SHARED_BLOCKS] = shared;
        row[KV_TRACE_CACHE_BYTES] = (int64_t)s.blocks.size() * block_bytes;
        row[KV_TRACE_REORDER_SRC] = s.reorder_src;
    }
    if (count) *count = (int)ids.size();
    return KV_OK;
}

int kv_slot_mapping(const int32_t* block_tables, int max_blocks, const int64_t* positions, int n,
                    int64_t* slot_mapping)
{
    if (n < 0 || max_blocks <= 0) return KV_ERR_INVALID_ARG;
    if (n > 0 && (!block_tables || !positions || !slot_mapping)) return KV_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
        int64_t pos = positions[i];
        if (pos < 0) {
            slot_mapping[i] = -1;
            continue;
        }
        int64_t bi = pos / KV_BLOCK_SIZE;
        if (bi >= max_blocks) return KV_ERR_INVALID_ARG;
        int32_t blk = block_tables[(int64_t)i * max_blocks + bi];
        if (blk < 0) return KV_ERR_INVALID_ARG;
        slot_mapping[i] = (int64_t)blk * KV_BLOCK_SIZE + pos % KV_BLOCK_SIZE;
    }
    return KV_OK;
}

// Prefix chunks from block tables ("KV cache complete guide", sections "(3)
// Prefix Caching" and "(4) PagedAttention": requests with a common system
// prompt hold the same physical blocks).  Groups by first block id, measures
// each member's common run with the group's longest member, orders members
// by that run and cuts them into chunks whose query rows fit one 16-row tile.
int kv_prefix_chunks(const int32_t* block_tables, int max_blocks_per_seq,
                     const int32_t* context_lens, int num_seqs, int group_size, int min_blocks,
                     int32_t* chunks, int32_t* seq_chunk, int* num_chunks)
{
    if (!num_chunks || num_seqs < 0 || max_blocks_per_seq <= 0 || group_size < 1 ||
        group_size > 8 || min_blocks < 1)
        return KV_ERR_INVALID_ARG;
    *num_chunks = 0;
    if (num_seqs == 0) return KV_OK;
    if (!block_tables || !context_lens || !chunks || !seq_chunk) return KV_ERR_INVALID_ARG;
    const int per_chunk = std::min(KV_PREFIX_MAX_ROWS / group_size, KV_PREFIX_MAX_MEMBERS);
    const int32_t* bt = block_tables;
    // full blocks before each sequence's new token (position L-1)
    std::vector<int> usable(num_seqs, 0);
    for (int s = 0; s < num_seqs; ++s) {
        seq_chunk[s] = -1;
        const int L = context_lens[s];
        if (L < 1) continue;
        usable[s] = std::min((L - 1) / KV_BLOCK_SIZE, max_blocks_per_seq);
    }
    // groups keyed by first block id, in order of first appearance
    std::map<int32_t, int> key_to_group;
    std::vector<std::vector<int>> groups;
    for (int s = 0; s < num_seqs; ++s) {
        if (usable[s] < min_blocks) continue;
        const int32_t first = bt[(int64_t)s * max_blocks_per_seq];
        if (first < 0) continue;
        auto it = key_to_group.find(first);
        if (it == key_to_group.end()) {
            key_to_group.emplace(first, (int)groups.size());
            groups.push_back({s});
        } else {
            groups[it->second].push_back(s);
        }
    }
    int nc = 0;
    for (const auto& gm : groups) {
        if (gm.size() < 2) continue;
        // the member with the most full blocks before its new token (the
        // first such) leads: every other member's run is measured on its row
        int lead = gm[0];
        for (int s : gm)
            if (usable[s] > usable[lead]) lead = s;
        const int32_t* lrow = bt + (int64_t)lead * max_blocks_per_seq;
        std::vector<std::pair<int, int>> run;    // (shared run, sequence)
        for (int s : gm) {
            const int32_t* row = bt + (int64_t)s * max_blocks_per_seq;
            const int cap = std::min(usable[s], usable[lead]);
            int r = 0;
            while (r < cap && row[r] == lrow[r] && row[r] >= 0) ++r;
            run.emplace_back(r, s);
        }
        std::stable_sort(run.begin(), run.end(), [](const std::pair<int, int>& a,
                                                    const std::pair<int, int>& b) {
            return a.first > b.first;
        });
        for (size_t i0 = 0; i0 < run.size(); i0 += per_chunk) {
            const size_t i1 = std::min(run.size(), i0 + (size_t)per_chunk);
            const int m = (int)(i1 - i0);
            const int P = run[i1 - 1].first;
            if (m < 2 || P < min_blocks) continue;
            int32_t* row = chunks + (int64_t)nc * KV_PREFIX_CHUNK_INTS;
            row[0] = P;
            row[1] = m;
            for (int k = 0; k < KV_PREFIX_MAX_MEMBERS; ++k)
                row[2 + k] = k < m ? run[i0 + k].second : -1;
            for (int k = 0; k < m; ++k) seq_chunk[run[i0 + k].second] = (nc << 4) | k;
            ++nc;
        }
    }
    *num_chunks = nc;
    return KV_OK;
}

const char* kv_version(void) { return "pagedkv 0.1 sm_103a"; }

}  // extern "C"

namespace pkv {

// Shared-prefix decoding trades a costlier kernel (two row tiles of state)
// for fewer bytes.  Whether it pays depends on the fraction f of the step's
// block reads the chunks save and on how many (sequence, KV head) pairs the
// step has against the split kernel's resident warps W.  Measured on GB300
// (fused step, 32 query / 8 KV heads, d128, W = 1216; groups of 8 sequences
// sharing a prompt of 32-256 blocks, lengths 4200-8192; f 6-50 %):
//   128 pairs: slower at every f (0.83-0.92x);
//   256 pairs: even at f = 6 % and 25 %, slower at 13 %, faster from 38 %
//              (1.10x; 1.22x at 51 %);
//   512 and 1024 pairs: faster at every f >= 6 % (1.02-1.77x);
//   2048 pairs: faster from f = 7.6 %, even at 3 %, slower at 5 % with
//              lengths spread over 16-32768.
// With few pairs the members of a group read their shared blocks close
// together and the plain kernel finds most of them in L2.  The rule: chunks
// when 5 pairs >= 2 W and f >= 6 %, or when 5 pairs >= W and f >= 30 %.
constexpr double kPrefixMinSavedFraction = 0.06;
constexpr double kPrefixMinSavedFractionFewPairs = 0.30;

int prefix_plan_host(const int32_t* block_tables, int max_blocks_per_seq,
                     const int32_t* context_lens, int num_seqs, int group_size,
                     int num_kv_heads, int resident_warps, int32_t* chunks, int32_t* seq_chunk,
                     int* num_chunks)
{
    if (!num_chunks || num_seqs < 0 || num_kv_heads < 1 || resident_warps < 1 ||
        group_size < 1)
        return KV_ERR_INVALID_ARG;
    *num_chunks = 0;
    if (num_seqs == 0) return KV_OK;
    if (!block_tables || !context_lens || !chunks || !seq_chunk || max_blocks_per_seq <= 0)
        return KV_ERR_INVALID_ARG;
    if (2 * group_size > KV_PREFIX_MAX_ROWS) {      // no chunks for groups above 8 rows
        for (int s = 0; s < num_seqs; ++s) seq_chunk[s] = -1;
        return KV_OK;
    }
    int nc = 0;
    if (int rc = kv_prefix_chunks(block_tables, max_blocks_per_seq, context_lens, num_seqs,
                                  group_size, 1, chunks, seq_chunk, &nc))
        return rc;
    if (nc == 0) return KV_OK;
    long long saved = 0, total = 0;
    for (int c = 0; c < nc; ++c) {
        const int32_t* row = chunks + (int64_t)c * KV_PREFIX_CHUNK_INTS;
        saved += (long long)row[0] * (row[1] - 1);
    }
    for (int s = 0; s < num_seqs; ++s) {
        const int L = std::min(std::max(context_lens[s], 0), max_blocks_per_seq * KV_BLOCK_SIZE);
        total += (L + KV_BLOCK_SIZE - 1) / KV_BLOCK_SIZE;
    }
    const long long pairs = (long long)num_seqs * num_kv_heads;
    const double f_min = 5 * pairs >= 2LL * resident_warps ? kPrefixMinSavedFraction
                         : 5 * pairs >= (long long)resident_warps ? kPrefixMinSavedFractionFewPairs
                                                                  : 2.0;   // never
    if ((double)saved >= f_min * (double)total) {
        *num_chunks = nc;
        return KV_OK;
    }
    for (int s = 0; s < num_seqs; ++s) seq_chunk[s] = -1;
    return KV_OK;
}

}  // namespace pkv
