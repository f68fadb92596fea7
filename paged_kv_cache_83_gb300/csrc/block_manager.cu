// block_manager.cu: the host block manager of the paged KV cache (C ABI in include/pa.h).
//
// Source: "nano-vLLM Part 4", sections 2 and 3 (the BlockManager's block IDs, reference counts and
// prefix-hash metadata; an exact full-block prefix cache; newly complete blocks hashed after each
// step; blocks freed when a sequence finishes); smzdm nano-vLLM deep dive, "调度与内存" (fixed-size
// blocks, reference counts, prefix cache for shared system prompts, preemption that frees blocks
// and keeps the tokens); "mini-vLLM" (a preallocated pool, an O(1) free-list allocator, a block
// table per sequence).
//
// Host code only: no GPU work. The structures:
//   * free blocks in a first-in first-out queue, kept as an intrusive doubly linked list over the
//     block ids, so a cached block that is reused can leave the middle of the queue in O(1);
//   * a full block is identified by its parent (the block before it when it was filled, as
//     (block id, generation), or the root) and its own tokens; a block taken from the free queue
//     for new content starts a new generation, which makes every cached block after it
//     unreachable. A match on (parent, tokens) is therefore a match on the whole prefix;
//   * the cache maps (parent, 64-bit hash of the block's tokens) to the most recently filled block
//     with that key; a hit is accepted only if the stored tokens are equal, so a hash collision
//     can cost a hit but never give a wrong one.
#include <stdint.h>
#include <string.h>

#include <new>
#include <unordered_map>
#include <vector>

#include "pa.h"

namespace {

constexpr uint64_t kRoot = ~0ull;

struct CacheKey {
    uint64_t parent, hash;
    bool operator==(const CacheKey &o) const { return parent == o.parent && hash == o.hash; }
};

uint64_t mix64(uint64_t x) {  // SplitMix64 finaliser (Steele, Lea, Flood 2014)
    x += 0x9e3779b97f4a7c15ull;
    x = (x ^ (x >> 30)) * 0xbf58476d1ce4e5b9ull;
    x = (x ^ (x >> 27)) * 0x94d049bb133111ebull;
    return x ^ (x >> 31);
}

struct CacheKeyHash {
    size_t operator()(const CacheKey &k) const { return static_cast<size_t>(mix64(k.parent ^ mix64(k.hash))); }
};

struct Sequence {
    std::vector<int32_t> tokens;
    std::vector<int32_t> table;
};

}  // namespace

struct pa_block_manager {
    int N, bs, flags;
    // free queue: intrusive doubly linked list
    std::vector<int32_t> prev, next;
    std::vector<uint8_t> in_free;
    int head = -1, tail = -1, nfree = 0;
    std::vector<int32_t> ref;
    std::vector<uint32_t> gen;
    std::vector<uint8_t> cached;      // has a cache key
    std::vector<CacheKey> key;        // its key while cached
    std::vector<int32_t> content;     // [N][bs] the tokens of cached blocks
    std::unordered_map<CacheKey, int32_t, CacheKeyHash> cache;
    std::unordered_map<int64_t, Sequence> seqs;

    uint64_t node(int b) const {
        return b < 0 ? kRoot : (static_cast<uint64_t>(gen[b]) << 32) | static_cast<uint32_t>(b);
    }
    uint64_t token_hash(const int32_t *t) const {
        if (flags & PA_BM_DEGENERATE_HASH) return 0;
        uint64_t h = 0x6a09e667f3bcc908ull;
        for (int i = 0; i < bs; ++i) h = mix64(h ^ static_cast<uint32_t>(t[i]));
        return h;
    }
    void push_back(int b) {
        prev[b] = tail;
        next[b] = -1;
        if (tail >= 0) next[tail] = b; else head = b;
        tail = b;
        in_free[b] = 1;
        ++nfree;
    }
    void unlink(int b) {
        if (prev[b] >= 0) next[prev[b]] = next[b]; else head = next[b];
        if (next[b] >= 0) prev[next[b]] = prev[b]; else tail = prev[b];
        in_free[b] = 0;
        --nfree;
    }
    // the front free block, for new content: it leaves the cache and starts a new generation
    int take_free() {
        const int b = head;
        unlink(b);
        if (cached[b]) {
            auto it = cache.find(key[b]);
            if (it != cache.end() && it->second == b) cache.erase(it);
            cached[b] = 0;
        }
        ++gen[b];
        return b;
    }
    void cache_block(int b, int parent, const int32_t *t) {
        const CacheKey k{node(parent), token_hash(t)};
        key[b] = k;
        cached[b] = 1;
        memcpy(&content[static_cast<size_t>(b) * bs], t, sizeof(int32_t) * bs);
        cache[k] = b;
    }
    // the cached blocks that start this token sequence (never the block of its last token)
    void match(const int32_t *t, int n, std::vector<int32_t> &out) const {
        out.clear();
        int parent = -1;
        for (int i = 0; i < (n - 1) / bs; ++i) {
            const int32_t *bt = t + static_cast<size_t>(i) * bs;
            auto it = cache.find(CacheKey{node(parent), token_hash(bt)});
            if (it == cache.end()) break;
            const int b = it->second;
            if (memcmp(&content[static_cast<size_t>(b) * bs], bt, sizeof(int32_t) * bs) != 0) break;
            out.push_back(b);
            parent = b;
        }
    }
    long long blocks_needed(const std::vector<int32_t> &m, int n) const {
        long long need = (static_cast<long long>(n) + bs - 1) / bs - static_cast<long long>(m.size());
        for (int b : m)
            if (ref[b] == 0) ++need;
        return need;
    }
};

extern "C" {

pa_block_manager *pa_bm_create(int num_blocks, int block_size, int flags) {
    if (num_blocks < 1 || block_size < 1 || (flags & ~PA_BM_DEGENERATE_HASH)) return nullptr;
    pa_block_manager *m = new (std::nothrow) pa_block_manager();
    if (!m) return nullptr;
    try {
        m->N = num_blocks;
        m->bs = block_size;
        m->flags = flags;
        m->prev.assign(num_blocks, -1);
        m->next.assign(num_blocks, -1);
        m->in_free.assign(num_blocks, 0);
        m->ref.assign(num_blocks, 0);
        m->gen.assign(num_blocks, 0);
        m->cached.assign(num_blocks, 0);
        m->key.assign(num_blocks, CacheKey{0, 0});
        m->content.assign(static_cast<size_t>(num_blocks) * block_size, 0);
        for (int b = 0; b < num_blocks; ++b) m->push_back(b);
    } catch (...) {
        delete m;
        return nullptr;
    }
    return m;
}

void pa_bm_destroy(pa_block_manager *m) { delete m; }

int pa_bm_num_free(const pa_block_manager *m) { return m ? m->nfree : PA_BM_ERR_ARG; }

int pa_bm_can_allocate(const pa_block_manager *m, const int32_t *tokens, int n) {
    if (!m || !tokens || n < 1) return PA_BM_ERR_ARG;
    std::vector<int32_t> matched;
    m->match(tokens, n, matched);
    return m->blocks_needed(matched, n) <= m->nfree ? 1 : 0;
}

int pa_bm_allocate(pa_block_manager *m, int64_t seq, const int32_t *tokens, int n) {
    if (!m || !tokens || n < 1) return PA_BM_ERR_ARG;
    if (m->seqs.count(seq)) return PA_BM_ERR_SEQ_EXISTS;
    std::vector<int32_t> matched;
    m->match(tokens, n, matched);
    if (m->blocks_needed(matched, n) > m->nfree) return PA_BM_ERR_NO_BLOCKS;
    Sequence s;
    s.tokens.assign(tokens, tokens + n);
    const int bs = m->bs;
    const int total = static_cast<int>((static_cast<long long>(n) + bs - 1) / bs);
    s.table.reserve(total);
    for (int b : matched) {
        if (m->ref[b] == 0) m->unlink(b);
        ++m->ref[b];
        s.table.push_back(b);
    }
    int parent = matched.empty() ? -1 : matched.back();
    for (int i = static_cast<int>(matched.size()); i < total; ++i) {
        const int b = m->take_free();
        m->ref[b] = 1;
        if (static_cast<long long>(i + 1) * bs <= n) m->cache_block(b, parent, tokens + static_cast<size_t>(i) * bs);
        s.table.push_back(b);
        parent = b;
    }
    m->seqs.emplace(seq, std::move(s));
    return static_cast<int>(matched.size()) * bs;
}

int64_t pa_bm_append(pa_block_manager *m, int64_t seq, int32_t token) {
    if (!m) return PA_BM_ERR_ARG;
    auto it = m->seqs.find(seq);
    if (it == m->seqs.end()) return PA_BM_ERR_NO_SEQ;
    Sequence &s = it->second;
    const int bs = m->bs;
    const long long n = static_cast<long long>(s.tokens.size());
    if (n >= INT32_MAX) return PA_BM_ERR_ARG;
    if (n % bs == 0) {
        if (m->nfree == 0) return PA_BM_ERR_NO_BLOCKS;
        const int b = m->take_free();
        m->ref[b] = 1;
        s.table.push_back(b);
    }
    s.tokens.push_back(token);
    const size_t i = static_cast<size_t>(n / bs);
    const int blk = s.table[i];
    if ((n + 1) % bs == 0)
        m->cache_block(blk, i > 0 ? s.table[i - 1] : -1, s.tokens.data() + i * bs);
    return static_cast<int64_t>(blk) * bs + n % bs;
}

int pa_bm_release(pa_block_manager *m, int64_t seq) {
    if (!m) return PA_BM_ERR_ARG;
    auto it = m->seqs.find(seq);
    if (it == m->seqs.end()) return PA_BM_ERR_NO_SEQ;
    const std::vector<int32_t> &t = it->second.table;
    for (size_t k = t.size(); k-- > 0;) {
        const int b = t[k];
        if (--m->ref[b] == 0) m->push_back(b);
    }
    m->seqs.erase(it);
    return 0;
}

int pa_bm_block_table(const pa_block_manager *m, int64_t seq, int32_t *out, int cap) {
    if (!m || cap < 0 || (cap > 0 && !out)) return PA_BM_ERR_ARG;
    auto it = m->seqs.find(seq);
    if (it == m->seqs.end()) return PA_BM_ERR_NO_SEQ;
    const std::vector<int32_t> &t = it->second.table;
    const int n = static_cast<int>(t.size());
    for (int k = 0; k < n && k < cap; ++k) out[k] = t[k];
    return n;
}

int pa_bm_num_tokens(const pa_block_manager *m, int64_t seq) {
    if (!m) return PA_BM_ERR_ARG;
    auto it = m->seqs.find(seq);
    return it == m->seqs.end() ? PA_BM_ERR_NO_SEQ : static_cast<int>(it->second.tokens.size());
}

int pa_bm_refcount(const pa_block_manager *m, int block) {
    if (!m || block < 0 || block >= m->N) return PA_BM_ERR_ARG;
    return m->ref[block];
}

}  // extern "C"
