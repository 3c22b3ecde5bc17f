// block_manager.cpp -- host-side paged KV block manager with chained-hash prefix caching.
//
// "AMD ATOM inference engine" (itsolotime.com), section 5.1: the KV cache is a pool of fixed-size
// blocks (16 tokens); each sequence keeps a block_table of the blocks it occupies; a Block has
// block_id, ref_count, hash (-1 when unset) and token_ids, reset() starts a block at ref_count 1.
// Section 5.2: prefix caching identifies a full block by xxhash64 over its token ids chained with
// the previous block's hash (the previous hash as 8 little-endian bytes, then the token ids as
// int64 bytes), so identical token blocks under different prefixes get different hashes.
// "LLM Primer VI, Chapter 8", section 8.1: blocks shared through reference counts.
//
// This is the step before the decode path: it turns sequences into the block_tables,
// context_lens and slot_mapping arrays the kernels take. Host state only (the caller owns the
// handle); not thread-safe. Free blocks are handed out first-in first-out, starting from block 0;
// a freed block keeps its hash and tokens, so a later prompt with the same prefix can take it back
// from the free list until it is reused for something else.
#include <cstdint>
#include <cstring>
#include <list>
#include <new>
#include <unordered_map>
#include <vector>

#include "pkv.h"

namespace {

// ---- XXH64 (the published xxHash 64-bit algorithm, seed 0 here) ----------------------------
constexpr uint64_t kP1 = 0x9E3779B185EBCA87ull, kP2 = 0xC2B2AE3D27D4EB4Full,
                   kP3 = 0x165667B19E3779F9ull, kP4 = 0x85EBCA77C2B2AE63ull,
                   kP5 = 0x27D4EB2F165667C5ull;

inline uint64_t rotl64(uint64_t x, int r) { return (x << r) | (x >> (64 - r)); }
inline uint64_t rd64(const uint8_t* p) {
    uint64_t v = 0;
    for (int i = 7; i >= 0; --i) v = (v << 8) | p[i];  // little-endian regardless of the host
    return v;
}
inline uint32_t rd32(const uint8_t* p) {
    return (uint32_t)p[0] | (uint32_t)p[1] << 8 | (uint32_t)p[2] << 16 | (uint32_t)p[3] << 24;
}
inline uint64_t xround(uint64_t acc, uint64_t in) { return rotl64(acc + in * kP2, 31) * kP1; }
inline uint64_t xmerge(uint64_t acc, uint64_t v) { return (acc ^ xround(0, v)) * kP1 + kP4; }

uint64_t xxh64(const uint8_t* p, size_t len, uint64_t seed) {
    const uint8_t* end = p + len;
    uint64_t h;
    if (len >= 32) {
        uint64_t v1 = seed + kP1 + kP2, v2 = seed + kP2, v3 = seed, v4 = seed - kP1;
        for (; p + 32 <= end; p += 32) {
            v1 = xround(v1, rd64(p));
            v2 = xround(v2, rd64(p + 8));
            v3 = xround(v3, rd64(p + 16));
            v4 = xround(v4, rd64(p + 24));
        }
        h = rotl64(v1, 1) + rotl64(v2, 7) + rotl64(v3, 12) + rotl64(v4, 18);
        h = xmerge(h, v1);
        h = xmerge(h, v2);
        h = xmerge(h, v3);
        h = xmerge(h, v4);
    } else {
        h = seed + kP5;
    }
    h += (uint64_t)len;
    for (; p + 8 <= end; p += 8) h = rotl64(h ^ xround(0, rd64(p)), 27) * kP1 + kP4;
    if (p + 4 <= end) {
        h = rotl64(h ^ (uint64_t)rd32(p) * kP1, 23) * kP2 + kP3;
        p += 4;
    }
    for (; p < end; ++p) h = rotl64(h ^ (uint64_t)(*p) * kP5, 11) * kP1;
    h ^= h >> 33;
    h *= kP2;
    h ^= h >> 29;
    h *= kP3;
    h ^= h >> 32;
    return h;
}

// Chained block hash: xxh64(prefix as 8 LE bytes if prefix != -1, then the tokens as int64 LE).
uint64_t block_hash(const int64_t* tokens, int n, int64_t prefix) {
    std::vector<uint8_t> buf;
    buf.reserve(8 + 8 * (size_t)n);
    auto put64 = [&](uint64_t v) {
        for (int i = 0; i < 8; ++i) buf.push_back((uint8_t)(v >> (8 * i)));
    };
    if (prefix != -1) put64((uint64_t)prefix);
    for (int i = 0; i < n; ++i) put64((uint64_t)tokens[i]);
    return xxh64(buf.data(), buf.size(), 0);
}

struct Block {
    int ref_count = 0;
    bool has_hash = false;
    uint64_t hash = 0;
    std::vector<int64_t> token_ids;  // the tokens of a full, hashed block
};

struct Sequence {
    std::vector<int32_t> table;
    std::vector<int64_t> tokens;
    bool last_full_hashed = false;  // hash of the last full block, for chaining
    uint64_t last_hash = 0;
};

}  // namespace

struct pkv_block_manager {
    int num_blocks, block_size;
    bool prefix_cache;
    std::vector<Block> blocks;
    std::list<int32_t> free_ids;                        // FIFO: take from the front
    std::vector<std::list<int32_t>::iterator> free_pos;  // where each free block sits in it
    std::unordered_map<uint64_t, int32_t> cached;  // hash -> block id
    std::unordered_map<int64_t, Sequence> seqs;

    void push_free(int32_t id) {
        free_ids.push_back(id);
        free_pos[id] = std::prev(free_ids.end());
    }
    int take_free_block() {  // front of the free list, forgetting what it cached
        const int32_t id = free_ids.front();
        free_ids.pop_front();
        free_pos[id] = free_ids.end();
        Block& blk = blocks[id];
        if (blk.has_hash) {
            auto it = cached.find(blk.hash);
            if (it != cached.end() && it->second == id) cached.erase(it);
        }
        blk.ref_count = 1;  // one user, nothing cached
        blk.has_hash = false;
        blk.token_ids.clear();
        return id;
    }
    void remove_from_free(int32_t id) {  // a free block taken back by a prefix hit
        free_ids.erase(free_pos[id]);
        free_pos[id] = free_ids.end();
    }
    // a block of the sequence just became full: give it its chained hash and cache it
    void seal(Sequence& s, int32_t id, const int64_t* toks) {
        if (!prefix_cache) return;
        const uint64_t h = block_hash(toks, block_size, s.last_full_hashed ? (int64_t)s.last_hash : -1);
        Block& blk = blocks[id];
        blk.has_hash = true;
        blk.hash = h;
        blk.token_ids.assign(toks, toks + block_size);
        cached[h] = id;
        s.last_full_hashed = true;
        s.last_hash = h;
    }
};

extern "C" {

pkv_block_manager* pkv_bm_create(int num_blocks, int block_size, int enable_prefix_cache) {
    if (num_blocks <= 0 || block_size <= 0) return nullptr;
    pkv_block_manager* bm = new (std::nothrow) pkv_block_manager();
    if (!bm) return nullptr;
    bm->num_blocks = num_blocks;
    bm->block_size = block_size;
    bm->prefix_cache = enable_prefix_cache != 0;
    bm->blocks.resize((size_t)num_blocks);
    bm->free_pos.resize((size_t)num_blocks);
    for (int i = 0; i < num_blocks; ++i) bm->push_free(i);
    return bm;
}

void pkv_bm_destroy(pkv_block_manager* bm) { delete bm; }

int pkv_bm_num_free_blocks(const pkv_block_manager* bm) { return bm ? (int)bm->free_ids.size() : -1; }

int pkv_bm_ref_count(const pkv_block_manager* bm, int block_id) {
    if (!bm || block_id < 0 || block_id >= bm->num_blocks) return -1;
    return bm->blocks[block_id].ref_count;
}

uint64_t pkv_xxh64(const void* data, size_t len, uint64_t seed) {
    return xxh64(static_cast<const uint8_t*>(data), len, seed);
}

uint64_t pkv_block_hash(const int64_t* token_ids, int num_tokens, int64_t prefix_hash) {
    return block_hash(token_ids, num_tokens, prefix_hash);
}

int pkv_bm_can_allocate(const pkv_block_manager* bm, int num_tokens) {
    if (!bm || num_tokens < 0) return 0;
    const long long need = ((long long)num_tokens + bm->block_size - 1) / bm->block_size;
    return (long long)bm->free_ids.size() >= need;
}

pkv_status pkv_bm_allocate(pkv_block_manager* bm, int64_t seq_id, const int64_t* token_ids,
                           int num_tokens, int* num_cached_tokens) {
    if (!bm || num_tokens < 0 || (num_tokens > 0 && !token_ids) || bm->seqs.count(seq_id))
        return PKV_ERR_INVALID_ARG;
    if (!pkv_bm_can_allocate(bm, num_tokens)) return PKV_ERR_NO_BLOCKS;
    Sequence s;
    int cached_tokens = 0;
    const int bs = bm->block_size;
    for (int i = 0; i * bs < num_tokens; ++i) {
        const int n = num_tokens - i * bs < bs ? num_tokens - i * bs : bs;
        const int64_t* toks = token_ids + (size_t)i * bs;
        int32_t id = -1;
        if (n == bs && bm->prefix_cache) {
            const uint64_t h = block_hash(toks, bs, s.last_full_hashed ? (int64_t)s.last_hash : -1);
            auto it = bm->cached.find(h);
            if (it != bm->cached.end() &&
                std::memcmp(bm->blocks[it->second].token_ids.data(), toks, sizeof(int64_t) * bs) == 0) {
                id = it->second;  // prefix hit: share the block
                Block& blk = bm->blocks[id];
                if (blk.ref_count == 0) bm->remove_from_free(id);
                blk.ref_count += 1;
                cached_tokens += bs;
                s.last_full_hashed = true;
                s.last_hash = h;
            }
        }
        if (id < 0) {
            id = bm->take_free_block();
            if (n == bs) bm->seal(s, id, toks);
        }
        s.table.push_back(id);
    }
    s.tokens.assign(token_ids, token_ids + num_tokens);
    bm->seqs.emplace(seq_id, std::move(s));
    if (num_cached_tokens) *num_cached_tokens = cached_tokens;
    return PKV_OK;
}

// Blocks an append of k tokens takes: those past the table's end, plus one when the tail block is
// partly filled and also referenced by another sequence (a fork), which is copied first.
static long long blocks_for_append(const pkv_block_manager* bm, const Sequence& s, int k) {
    const long long n = (long long)s.tokens.size();
    long long need = (n + k + bm->block_size - 1) / bm->block_size - (long long)s.table.size();
    if (k > 0 && n % bm->block_size != 0 && bm->blocks[s.table.back()].ref_count > 1) need += 1;
    return need;
}

int pkv_bm_can_append(const pkv_block_manager* bm, int64_t seq_id, int num_new_tokens) {
    if (!bm || num_new_tokens < 0) return 0;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return 0;
    const long long need = blocks_for_append(bm, it->second, num_new_tokens);
    return need <= 0 || (long long)bm->free_ids.size() >= need;
}

pkv_status pkv_bm_append_cow(pkv_block_manager* bm, int64_t seq_id, const int64_t* new_token_ids,
                             int num_new_tokens, int64_t* slot_mapping, int32_t* copy_src_dst,
                             int* num_copies) {
    if (num_copies) *num_copies = 0;
    if (!bm || num_new_tokens < 0 || (num_new_tokens > 0 && !new_token_ids)) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
    Sequence& s = it->second;
    const int bs = bm->block_size;
    // a shared, partly filled tail block must be copied before the first new token lands in it
    const bool cow = num_new_tokens > 0 && s.tokens.size() % bs != 0 && bm->blocks[s.table.back()].ref_count > 1;
    if (cow && (!copy_src_dst || !num_copies)) return PKV_ERR_INVALID_ARG;
    if (!pkv_bm_can_append(bm, seq_id, num_new_tokens)) return PKV_ERR_NO_BLOCKS;
    if (cow) {
        const int32_t src = s.table.back();
        const int32_t dst = bm->take_free_block();
        bm->blocks[src].ref_count -= 1;  // still >= 1: another sequence keeps it
        s.table.back() = dst;
        copy_src_dst[0] = src;
        copy_src_dst[1] = dst;
        *num_copies = 1;
    }
    for (int k = 0; k < num_new_tokens; ++k) {
        const size_t pos = s.tokens.size();
        if (pos % bs == 0) s.table.push_back(bm->take_free_block());
        const int32_t id = s.table[pos / bs];
        if (slot_mapping) slot_mapping[k] = (int64_t)id * bs + (int64_t)(pos % bs);
        s.tokens.push_back(new_token_ids[k]);
        if (pos % bs == (size_t)bs - 1) bm->seal(s, id, s.tokens.data() + (pos + 1 - bs));
    }
    return PKV_OK;
}

pkv_status pkv_bm_append(pkv_block_manager* bm, int64_t seq_id, const int64_t* new_token_ids,
                         int num_new_tokens, int64_t* slot_mapping) {
    return pkv_bm_append_cow(bm, seq_id, new_token_ids, num_new_tokens, slot_mapping, nullptr, nullptr);
}

pkv_status pkv_bm_fork(pkv_block_manager* bm, int64_t parent_id, int64_t child_id) {
    if (!bm || parent_id == child_id || bm->seqs.count(child_id)) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(parent_id);
    if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
    Sequence child = it->second;  // same table, tokens and hash-chain link
    for (int32_t id : child.table) bm->blocks[id].ref_count += 1;
    bm->seqs.emplace(child_id, std::move(child));
    return PKV_OK;
}

pkv_status pkv_bm_free(pkv_block_manager* bm, int64_t seq_id) {
    if (!bm) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
    const std::vector<int32_t>& t = it->second.table;
    for (auto r = t.rbegin(); r != t.rend(); ++r) {  // tail first: the prefix stays cached longest
        Block& blk = bm->blocks[*r];
        if (--blk.ref_count == 0) bm->push_free(*r);
    }
    bm->seqs.erase(it);
    return PKV_OK;
}

int pkv_bm_context_len(const pkv_block_manager* bm, int64_t seq_id) {
    if (!bm) return -1;
    auto it = bm->seqs.find(seq_id);
    return it == bm->seqs.end() ? -1 : (int)it->second.tokens.size();
}

pkv_status pkv_bm_batch_tables(const pkv_block_manager* bm, const int64_t* seq_ids, int num_seqs,
                               int max_blocks_per_seq, int32_t* block_tables,
                               int32_t* context_lens) {
    if (!bm || num_seqs < 0 || max_blocks_per_seq <= 0 || (num_seqs > 0 && (!seq_ids || !block_tables)))
        return PKV_ERR_INVALID_ARG;
    for (int b = 0; b < num_seqs; ++b) {
        auto it = bm->seqs.find(seq_ids[b]);
        if (it == bm->seqs.end() || (int)it->second.table.size() > max_blocks_per_seq)
            return PKV_ERR_INVALID_ARG;
        const std::vector<int32_t>& t = it->second.table;
        int32_t* row = block_tables + (size_t)b * max_blocks_per_seq;
        for (int j = 0; j < max_blocks_per_seq; ++j) row[j] = j < (int)t.size() ? t[j] : -1;
        if (context_lens) context_lens[b] = (int32_t)it->second.tokens.size();
    }
    return PKV_OK;
}

}  // extern "C"
