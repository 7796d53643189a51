// Host block manager: physical-block allocation, reference counts,
// copy-on-write and automatic prefix caching for the paged KV pool.
//
// Follows the page "vLLM PagedAttention chuyen sau" (locionic.com):
//   - "Tuong tu phan trang bo nho ao": a sequence's KV lives in fixed-size
//     logical blocks mapped through its block table to physical blocks
//     anywhere in the pool; blocks may be shared; a growing sequence gets new
//     physical blocks on demand, without copying what it already has;
//   - "Co che APC": a prefix tree of KV blocks; a new request is matched
//     against it and the physical blocks of the matched prefix are linked
//     straight into its block table; a sequence that diverges from a shared
//     block copies that block first (copy-on-write);
//   - "Danh gia ty le truy cap APC": the hit rate is the share of tokens whose
//     KV blocks were reused from an existing prefix;
//   - FAQ item 5: under memory pressure blocks are evicted least recently
//     used first.
// Readings where the page is loose: the tree is kept at block granularity
// (a node is one full block of block_size token ids, keyed by those ids),
// because only whole physical blocks can be shared; a partially filled block
// is never in the tree.  Blocks whose reference count drops to zero stay in
// the tree, reusable, until evicted; eviction takes the least recently
// released leaf, so no cached block loses its parent.
//
// Not thread-safe: one owner drives a manager.  The manager only does
// bookkeeping; the caller moves the data (pa_copy_blocks for the copy pairs,
// pa_reshape_and_cache for the returned slots) before the next kernel reads
// the blocks.

#include <cstdint>
#include <list>
#include <map>
#include <memory>
#include <unordered_map>
#include <vector>

#include "../../include/pa.h"

namespace {

struct Node {
    int32_t block = -1;
    Node *parent = nullptr;
    std::vector<int32_t> tokens;                               // the block's token ids
    std::map<std::vector<int32_t>, std::unique_ptr<Node>> children;
    std::list<Node *>::iterator lru;                           // valid while released
    bool released = false;
};

struct Seq {
    std::vector<int32_t> blocks;
    int64_t len = 0;
    std::vector<int32_t> tail;  // token ids in the last, partially filled block
    Node *node = nullptr;       // tree node of the last full block, if every full block is in the tree
    bool chained = true;        // all full blocks so far are tree nodes (so new full blocks can join)
};

}  // namespace

struct pa_block_manager {
    int num_blocks = 0, block_size = 0;
    bool prefix_cache = false;
    std::vector<int32_t> refc;
    std::vector<int32_t> free_list;
    std::vector<Node *> node_of;  // tree node holding each block, or null
    Node root;
    std::list<Node *> lru;        // released cached blocks, least recently released first
    std::unordered_map<int64_t, Seq> seqs;
    long long query_tokens = 0, hit_tokens = 0, evictions = 0, cow_copies = 0;

    // a block for new data: from the free list, else by evicting the least
    // recently released cached leaf; -1 if neither exists
    int32_t alloc() {
        if (!free_list.empty()) {
            const int32_t b = free_list.back();
            free_list.pop_back();
            refc[b] = 1;
            return b;
        }
        for (auto it = lru.begin(); it != lru.end(); ++it) {
            Node *n = *it;
            if (!n->children.empty()) continue;
            const int32_t b = n->block;
            lru.erase(it);
            node_of[b] = nullptr;
            ++evictions;
            auto &siblings = n->parent->children;
            siblings.erase(siblings.find(n->tokens));  // frees n
            refc[b] = 1;
            return b;
        }
        return -1;
    }

    void retain(int32_t b) {
        if (refc[b]++ == 0 && node_of[b] && node_of[b]->released) {
            lru.erase(node_of[b]->lru);
            node_of[b]->released = false;
        }
    }

    void release(int32_t b) {
        if (--refc[b] > 0) return;
        if (Node *n = node_of[b]) {
            n->lru = lru.insert(lru.end(), n);
            n->released = true;
        } else {
            free_list.push_back(b);
        }
    }

    // the sequence's last block just filled up: make it a tree node if its
    // whole prefix is in the tree and no node with these tokens exists yet
    void maybe_cache_full_block(Seq &s) {
        if (!prefix_cache || !s.chained) return;
        Node *parent = s.node ? s.node : &root;
        const int32_t b = s.blocks.back();
        auto it = parent->children.find(s.tail);
        if (it != parent->children.end() || node_of[b]) {
            // same content already cached under another block: this copy stays private
            s.chained = false;
            return;
        }
        auto n = std::make_unique<Node>();
        n->block = b;
        n->parent = parent;
        n->tokens = s.tail;
        Node *raw = n.get();
        parent->children.emplace(s.tail, std::move(n));
        node_of[b] = raw;
        s.node = raw;
    }
};

extern "C" {

pa_block_manager *pa_bm_create(int num_blocks, int block_size, int enable_prefix_cache) {
    if (num_blocks <= 0 || block_size <= 0) return nullptr;
    auto *m = new pa_block_manager();
    m->num_blocks = num_blocks;
    m->block_size = block_size;
    m->prefix_cache = enable_prefix_cache != 0;
    m->refc.assign(num_blocks, 0);
    m->node_of.assign(num_blocks, nullptr);
    m->free_list.reserve(num_blocks);
    // hand blocks out in increasing id order
    for (int b = num_blocks - 1; b >= 0; --b) m->free_list.push_back(b);
    return m;
}

void pa_bm_destroy(pa_block_manager *m) { delete m; }

int pa_bm_add_sequence(pa_block_manager *m, int64_t seq_id, const int32_t *tokens, int num_tokens,
                       int64_t *slots, int *num_cached_tokens) {
    if (!m || num_tokens < 0 || (num_tokens > 0 && (!tokens || !slots))) return PA_ERR_INVALID_ARG;
    if (m->seqs.count(seq_id)) return PA_ERR_INVALID_ARG;
    const int bs = m->block_size;
    Seq s;
    int cached = 0;
    if (m->prefix_cache) {
        // link the longest run of full blocks already in the prefix tree
        Node *node = &m->root;
        std::vector<int32_t> key(bs);
        while (cached + bs <= num_tokens) {
            key.assign(tokens + cached, tokens + cached + bs);
            auto it = node->children.find(key);
            if (it == node->children.end()) break;
            node = it->second.get();
            m->retain(node->block);
            s.blocks.push_back(node->block);
            cached += bs;
        }
        s.node = node == &m->root ? nullptr : node;
    }
    // fresh blocks for the rest, all taken before anything else changes so
    // that running out leaves the manager exactly as it was
    const int need = (num_tokens + bs - 1) / bs - (int)s.blocks.size();
    std::vector<int32_t> fresh;
    fresh.reserve(need > 0 ? need : 0);
    for (int k = 0; k < need; ++k) {
        const int32_t b = m->alloc();
        if (b < 0) {
            for (int32_t f : fresh) m->release(f);
            for (auto it = s.blocks.rbegin(); it != s.blocks.rend(); ++it) m->release(*it);
            return PA_ERR_NO_BLOCKS;
        }
        fresh.push_back(b);
    }
    for (int i = cached, k = 0; i < num_tokens; ++i) {
        if (i % bs == 0) s.blocks.push_back(fresh[k++]);
        s.tail.push_back(tokens[i]);
        slots[i] = (int64_t)s.blocks.back() * bs + i % bs;
        if ((i + 1) % bs == 0) {
            m->maybe_cache_full_block(s);
            s.tail.clear();
        }
    }
    for (int i = 0; i < cached && slots; ++i) slots[i] = -1;
    s.len = num_tokens;
    m->query_tokens += num_tokens;
    m->hit_tokens += cached;
    if (num_cached_tokens) *num_cached_tokens = cached;
    m->seqs.emplace(seq_id, std::move(s));
    return PA_OK;
}

int pa_bm_fork(pa_block_manager *m, int64_t parent_id, int64_t child_id) {
    if (!m) return PA_ERR_INVALID_ARG;
    auto it = m->seqs.find(parent_id);
    if (it == m->seqs.end() || m->seqs.count(child_id)) return PA_ERR_INVALID_ARG;
    Seq c = it->second;
    for (int32_t b : c.blocks) m->retain(b);
    m->seqs.emplace(child_id, std::move(c));
    return PA_OK;
}

int pa_bm_append_token(pa_block_manager *m, int64_t seq_id, int32_t token, int64_t *slot,
                       int64_t *copy_src, int64_t *copy_dst) {
    if (!m || !slot) return PA_ERR_INVALID_ARG;
    auto it = m->seqs.find(seq_id);
    if (it == m->seqs.end()) return PA_ERR_INVALID_ARG;
    Seq &s = it->second;
    const int bs = m->block_size;
    const int off = (int)(s.len % bs);
    int64_t src = -1, dst = -1;
    if (off == 0) {
        const int32_t b = m->alloc();
        if (b < 0) return PA_ERR_NO_BLOCKS;
        s.blocks.push_back(b);
    } else if (m->refc[s.blocks.back()] > 1) {
        // copy-on-write: the partial last block is shared; write into a private copy
        const int32_t b = m->alloc();
        if (b < 0) return PA_ERR_NO_BLOCKS;
        src = s.blocks.back();
        dst = b;
        m->release(s.blocks.back());
        s.blocks.back() = b;
        ++m->cow_copies;
    }
    *slot = (int64_t)s.blocks.back() * bs + off;
    if (copy_src) *copy_src = src;
    if (copy_dst) *copy_dst = dst;
    s.tail.push_back(token);
    ++s.len;
    if (s.len % bs == 0) {
        m->maybe_cache_full_block(s);
        s.tail.clear();
    }
    return PA_OK;
}

int pa_bm_free_sequence(pa_block_manager *m, int64_t seq_id) {
    if (!m) return PA_ERR_INVALID_ARG;
    auto it = m->seqs.find(seq_id);
    if (it == m->seqs.end()) return PA_ERR_INVALID_ARG;
    // last block first, so deeper cached blocks are evicted before their parents
    const auto &blocks = it->second.blocks;
    for (auto b = blocks.rbegin(); b != blocks.rend(); ++b) m->release(*b);
    m->seqs.erase(it);
    return PA_OK;
}

int pa_bm_block_table(const pa_block_manager *m, int64_t seq_id, int32_t *out, int max_blocks) {
    if (!m) return PA_ERR_INVALID_ARG;
    auto it = m->seqs.find(seq_id);
    if (it == m->seqs.end()) return PA_ERR_INVALID_ARG;
    const auto &blocks = it->second.blocks;
    if ((int64_t)blocks.size() > max_blocks || (!out && !blocks.empty())) return PA_ERR_OUT_OF_RANGE;
    for (size_t i = 0; i < blocks.size(); ++i) out[i] = blocks[i];
    return (int)blocks.size();
}

int64_t pa_bm_seq_len(const pa_block_manager *m, int64_t seq_id) {
    if (!m) return PA_ERR_INVALID_ARG;
    auto it = m->seqs.find(seq_id);
    return it == m->seqs.end() ? (int64_t)PA_ERR_INVALID_ARG : it->second.len;
}

int pa_bm_block_refcount(const pa_block_manager *m, int block) {
    if (!m || block < 0 || block >= m->num_blocks) return PA_ERR_INVALID_ARG;
    return m->refc[block];
}

int pa_bm_stats(const pa_block_manager *m, pa_bm_counters *out) {
    if (!m || !out) return PA_ERR_INVALID_ARG;
    out->num_blocks = m->num_blocks;
    out->free_blocks = (int)m->free_list.size();
    out->cached_free_blocks = (int)m->lru.size();
    out->used_blocks = m->num_blocks - out->free_blocks - out->cached_free_blocks;
    out->num_sequences = (int)m->seqs.size();
    out->query_tokens = m->query_tokens;
    out->hit_tokens = m->hit_tokens;
    out->evictions = m->evictions;
    out->cow_copies = m->cow_copies;
    return PA_OK;
}

}  // extern "C"
