// Host-side block manager of the paged KV cache (C ABI in include/pkv.h).
//
// "How does TensorRT-LLM work?", "The paged KV cache": the KV memory is one
// pool of equal blocks handed out one at a time when a request needs room; a
// small table keeps each request's blocks in order; a finished request's
// blocks go straight back to the free pool; requests that begin with the same
// text can point at the very same blocks (prefix reuse).
// "TensorRT-LLM, in depth", "In-flight batching and the scheduler": a running
// request that cannot get a block for its next token is paused; "The paged
// KV cache and block reuse": cached blocks are reused only for byte-identical
// token prefixes.
//
// Design:
//   * ref[b] counts the sequences whose table holds block b; a block with
//     ref 0 is on the free list.
//   * The free list is doubly linked: blocks are taken from the head and
//     returned to the tail, so a freed block that holds a complete, hashed
//     prefix stays matchable until it is reallocated (LRU eviction).
//   * A full block's identity is a 64-bit chain hash of the token ids of the
//     whole prefix up to and including it (FNV-1a over the parent hash and
//     the block's ids); the cache maps hash -> block.  Blocks written by
//     tokens without ids (generated tokens) are never hashed.
//   * Shared blocks are always full, so no sequence ever writes into a block
//     another sequence reads.
#include <cstdint>
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "pkv.h"

struct pkv_block_manager {
    struct Seq {
        std::vector<int32_t> blocks;
        int32_t len = 0;
        bool hashable = true;            // every token so far came with an id
        uint64_t chain = 0;              // hash of the full blocks so far
        std::vector<int32_t> open_ids;   // ids of the tokens in the partial last block
    };
    int32_t num_blocks = 0, bs = 0, max_blocks = 0;
    std::vector<int32_t> ref, prev, next;
    std::vector<uint8_t> hashed;
    std::vector<uint64_t> hash_of;
    int32_t head = -1, tail = -1, nfree = 0;
    std::unordered_map<uint64_t, int32_t> cache;
    std::unordered_map<int64_t, Seq> seqs;

    static uint64_t chain_hash(uint64_t parent, const int32_t* ids, int n) {
        uint64_t h = 1469598103934665603ull ^ parent;
        for (int i = 0; i < n; ++i) {
            uint32_t v = static_cast<uint32_t>(ids[i]);
            for (int k = 0; k < 4; ++k) {
                h ^= (v >> (8 * k)) & 0xFFu;
                h *= 1099511628211ull;
            }
        }
        return h ? h : 1;  // 0 marks "no parent"
    }
    void push_tail(int32_t b) {
        prev[b] = tail;
        next[b] = -1;
        if (tail >= 0) next[tail] = b; else head = b;
        tail = b;
        ++nfree;
    }
    void unlink(int32_t b) {
        if (prev[b] >= 0) next[prev[b]] = next[b]; else head = next[b];
        if (next[b] >= 0) prev[next[b]] = prev[b]; else tail = prev[b];
        prev[b] = next[b] = -1;
        --nfree;
    }
    bool on_free_list(int32_t b) const { return ref[b] == 0; }
    void forget_hash(int32_t b) {
        if (hashed[b]) {
            auto it = cache.find(hash_of[b]);
            if (it != cache.end() && it->second == b) cache.erase(it);
            hashed[b] = 0;
        }
    }
    int32_t take_free() {  // head of the free list, evicted from the cache
        const int32_t b = head;
        unlink(b);
        forget_hash(b);
        ref[b] = 1;
        return b;
    }
    void release(int32_t b) {
        if (--ref[b] == 0) push_tail(b);
    }
    int32_t blocks_for(int64_t tokens) const { return static_cast<int32_t>((tokens + bs - 1) / bs); }

    // Account for n tokens appended to s (ids may be null): hash blocks that
    // become full while the sequence is still hashable.
    void note_tokens(Seq& s, const int32_t* ids, int32_t n) {
        for (int32_t i = 0; i < n; ++i) {
            if (!ids) s.hashable = false;
            if (!s.hashable) continue;
            s.open_ids.push_back(ids[i]);
            if (static_cast<int32_t>(s.open_ids.size()) == bs) {
                const int32_t blk_index = (s.len + i) / bs;
                const int32_t b = s.blocks[blk_index];
                s.chain = chain_hash(s.chain, s.open_ids.data(), bs);
                s.open_ids.clear();
                if (!hashed[b] && cache.find(s.chain) == cache.end()) {
                    cache.emplace(s.chain, b);
                    hashed[b] = 1;
                    hash_of[b] = s.chain;
                }
            }
        }
    }
};

extern "C" {

pkv_status kv_block_manager_create(int32_t num_blocks, int32_t block_size, int32_t max_blocks_per_seq,
                                   const int32_t* free_order, pkv_block_manager** out) {
    if (!out || num_blocks < 1 || block_size < 1 || max_blocks_per_seq < 1) return PKV_ERR_INVALID_ARG;
    *out = nullptr;
    pkv_block_manager* m = new (std::nothrow) pkv_block_manager();
    if (!m) return PKV_ERR_INVALID_ARG;
    m->num_blocks = num_blocks;
    m->bs = block_size;
    m->max_blocks = max_blocks_per_seq;
    m->ref.assign(num_blocks, 0);
    m->prev.assign(num_blocks, -1);
    m->next.assign(num_blocks, -1);
    m->hashed.assign(num_blocks, 0);
    m->hash_of.assign(num_blocks, 0);
    std::vector<uint8_t> seen(num_blocks, 0);
    for (int32_t i = 0; i < num_blocks; ++i) {
        const int32_t b = free_order ? free_order[i] : i;
        if (b < 0 || b >= num_blocks || seen[b]) {
            delete m;
            return PKV_ERR_INVALID_ARG;  // not a permutation of the pool's ids
        }
        seen[b] = 1;
        m->push_tail(b);
    }
    *out = m;
    return PKV_OK;
}

void kv_block_manager_destroy(pkv_block_manager* m) { delete m; }

int32_t kv_bm_num_free(const pkv_block_manager* m) { return m ? m->nfree : -1; }

pkv_status kv_bm_add_sequence(pkv_block_manager* m, int64_t seq) {
    if (!m || m->seqs.count(seq)) return PKV_ERR_INVALID_ARG;
    m->seqs.emplace(seq, pkv_block_manager::Seq());
    return PKV_OK;
}

pkv_status kv_bm_free_sequence(pkv_block_manager* m, int64_t seq) {
    if (!m) return PKV_ERR_INVALID_ARG;
    auto it = m->seqs.find(seq);
    if (it == m->seqs.end()) return PKV_ERR_INVALID_ARG;
    for (int32_t b : it->second.blocks) m->release(b);
    m->seqs.erase(it);
    return PKV_OK;
}

pkv_status kv_bm_grow(pkv_block_manager* m, int64_t seq, int32_t n_tokens, const int32_t* token_ids,
                      int64_t* slots_out) {
    if (!m || n_tokens < 0) return PKV_ERR_INVALID_ARG;
    auto it = m->seqs.find(seq);
    if (it == m->seqs.end()) return PKV_ERR_INVALID_ARG;
    auto& s = it->second;
    const int64_t new_len = static_cast<int64_t>(s.len) + n_tokens;
    const int32_t need_total = m->blocks_for(new_len);
    if (need_total > m->max_blocks) return PKV_ERR_OUT_OF_BLOCKS;
    const int32_t need = need_total - static_cast<int32_t>(s.blocks.size());
    if (need > m->nfree) return PKV_ERR_OUT_OF_BLOCKS;
    for (int32_t i = 0; i < need; ++i) s.blocks.push_back(m->take_free());
    if (slots_out)
        for (int32_t i = 0; i < n_tokens; ++i) {
            const int64_t p = s.len + i;
            slots_out[i] = static_cast<int64_t>(s.blocks[p / m->bs]) * m->bs + p % m->bs;
        }
    m->note_tokens(s, token_ids, n_tokens);
    s.len = static_cast<int32_t>(new_len);
    return PKV_OK;
}

pkv_status kv_bm_decode_slots(pkv_block_manager* m, const int64_t* seq_ids, int32_t n, int64_t* slots_out,
                              int32_t* n_paused) {
    if (!m || n < 0 || (n > 0 && (!seq_ids || !slots_out))) return PKV_ERR_INVALID_ARG;
    int32_t paused = 0;
    for (int32_t i = 0; i < n; ++i) {
        if (!m->seqs.count(seq_ids[i])) return PKV_ERR_INVALID_ARG;
        const pkv_status st = kv_bm_grow(m, seq_ids[i], 1, nullptr, &slots_out[i]);
        if (st == PKV_ERR_OUT_OF_BLOCKS) {
            slots_out[i] = -1;  // paused: no block for its next token this step
            ++paused;
        } else if (st != PKV_OK) {
            return st;
        }
    }
    if (n_paused) *n_paused = paused;
    return PKV_OK;
}

pkv_status kv_bm_match_prefix(pkv_block_manager* m, int64_t seq, const int32_t* token_ids, int32_t n_tokens,
                              int32_t* reused_tokens_out) {
    if (!m || n_tokens < 0 || (n_tokens > 0 && !token_ids)) return PKV_ERR_INVALID_ARG;
    auto it = m->seqs.find(seq);
    if (it == m->seqs.end() || it->second.len != 0) return PKV_ERR_INVALID_ARG;
    auto& s = it->second;
    // whole blocks only, and never the token the caller still has to append
    const int32_t max_full = n_tokens > 0 ? (n_tokens - 1) / m->bs : 0;
    int32_t reused = 0;
    uint64_t h = 0;
    for (int32_t k = 0; k < max_full && k < m->max_blocks; ++k) {
        const uint64_t hk = pkv_block_manager::chain_hash(h, token_ids + static_cast<int64_t>(k) * m->bs, m->bs);
        auto c = m->cache.find(hk);
        if (c == m->cache.end()) break;
        const int32_t b = c->second;
        if (m->on_free_list(b)) {  // revive a cached free block
            m->unlink(b);
            m->ref[b] = 1;
        } else {
            ++m->ref[b];
        }
        s.blocks.push_back(b);
        h = hk;
        reused += m->bs;
    }
    s.len = reused;
    s.chain = h;
    if (reused_tokens_out) *reused_tokens_out = reused;
    return PKV_OK;
}

int32_t kv_bm_seq_len(const pkv_block_manager* m, int64_t seq) {
    if (!m) return -1;
    auto it = m->seqs.find(seq);
    return it == m->seqs.end() ? -1 : it->second.len;
}

pkv_status kv_bm_block_tables(const pkv_block_manager* m, const int64_t* seq_ids, int32_t n, int32_t width,
                              int32_t* tables_out, int32_t* lens_out) {
    if (!m || n < 0 || width < 1 || (n > 0 && !seq_ids)) return PKV_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n; ++i) {
        auto it = m->seqs.find(seq_ids[i]);
        if (it == m->seqs.end()) return PKV_ERR_INVALID_ARG;
        const auto& s = it->second;
        if (static_cast<int32_t>(s.blocks.size()) > width) return PKV_ERR_INVALID_ARG;
        if (tables_out) {
            int32_t* row = tables_out + static_cast<int64_t>(i) * width;
            for (int32_t k = 0; k < width; ++k) row[k] = k < static_cast<int32_t>(s.blocks.size()) ? s.blocks[k] : -1;
        }
        if (lens_out) lens_out[i] = s.len;
    }
    return PKV_OK;
}

int32_t kv_bm_free_list(const pkv_block_manager* m, int32_t* out, int32_t cap) {
    if (!m) return -1;
    int32_t k = 0;
    for (int32_t b = m->head; b >= 0; b = m->next[b]) {
        if (out && k < cap) out[k] = b;
        ++k;
    }
    return k;
}

int32_t kv_bm_block_ref(const pkv_block_manager* m, int32_t block) {
    if (!m || block < 0 || block >= m->num_blocks) return -1;
    return m->ref[block];
}

pkv_status kv_bm_check(const pkv_block_manager* m) {
    if (!m) return PKV_ERR_INVALID_ARG;
    std::vector<int32_t> count(m->num_blocks, 0);
    for (const auto& kv : m->seqs) {
        const auto& s = kv.second;
        if (static_cast<int32_t>(s.blocks.size()) != m->blocks_for(s.len)) return PKV_ERR_INCONSISTENT;
        for (int32_t b : s.blocks) ++count[b];
    }
    int32_t free_seen = 0;
    for (int32_t b = m->head, last = -1; b >= 0; last = b, b = m->next[b]) {
        if (m->prev[b] != last || m->ref[b] != 0) return PKV_ERR_INCONSISTENT;
        if (++free_seen > m->num_blocks) return PKV_ERR_INCONSISTENT;
    }
    if (free_seen != m->nfree) return PKV_ERR_INCONSISTENT;
    for (int32_t b = 0; b < m->num_blocks; ++b)
        if (count[b] != m->ref[b]) return PKV_ERR_INCONSISTENT;
    for (const auto& kv : m->cache)
        if (!m->hashed[kv.second] || m->hash_of[kv.second] != kv.first) return PKV_ERR_INCONSISTENT;
    return PKV_OK;
}

}  // extern "C"
