// Host block manager: physical block allocation, reference counts,
// copy-on-write and a prefix index for the paged KV cache.
//
// The paging scheme follows the PagedAttention description (ainews
// "PagedAttention": a sequence's logical blocks map to physical blocks that
// are allocated on demand and need not be contiguous; sequences may share
// physical blocks, and a shared block that must change is copied first) and
// the runtime page's "Paging" and "Prefix caching" sections (full blocks of
// a common prompt prefix are reused by later requests; unreferenced cached
// blocks are evicted least recently used first).  What it produces are the
// inputs of the kernels: block tables, context lengths, slot mappings and
// copy-on-write (src, dst) pairs.  Host memory only; no CUDA call.
#include <stdint.h>
#include <string.h>

#include <array>
#include <set>
#include <unordered_map>
#include <utility>
#include <vector>

#include "pkv.h"

namespace pkv {
int fail(int code, const char *fmt, ...);
}

namespace {

constexpr int kBs = PKV_BLOCK_SIZE;

// splitmix64 finaliser: a well-mixed 64-bit function of its input
uint64_t mix64(uint64_t x) {
    x += 0x9e3779b97f4a7c15ull;
    x = (x ^ (x >> 30)) * 0xbf58476d1ce4e5b9ull;
    x = (x ^ (x >> 27)) * 0x94d049bb133111ebull;
    return x ^ (x >> 31);
}

// Chain hash of a full block: its 16 token ids and the previous block's hash.
uint64_t block_hash(uint64_t prev, const int32_t *tok) {
    uint64_t h = mix64(prev ^ 0x5851f42d4c957f2dull);
    for (int i = 0; i < kBs; i++) h = mix64(h ^ (uint32_t)tok[i]);
    return h;
}

struct Block {
    int ref = 0;              // sequences whose table holds this block
    int ntok = 0;             // tokens written (rows in use)
    bool registered = false;  // in the prefix index (full, content known)
    uint64_t hash = 0;        // chain hash (registered blocks)
    uint64_t last_use = 0;    // for least-recently-used eviction
    uint32_t gen = 0;         // times this block has been handed out
    // registered blocks: the block before this one in the chain it was
    // registered under (-1 for a first block) and that block's gen then
    int32_t parent = -1;
    uint32_t parent_gen = 0;
    std::array<int32_t, kBs> tok{};
};

struct Seq {
    std::vector<int32_t> blocks;
    int len = 0;
    uint64_t tail_hash = 0;  // chain hash of the last full block (0 before the first)
};

class BlockManager {
  public:
    BlockManager(int num_blocks, int max_blocks, bool prefix)
        : blocks_(num_blocks), max_blocks_(max_blocks), prefix_(prefix) {
        free_.reserve(num_blocks);
        for (int b = num_blocks - 1; b >= 0; b--) free_.push_back(b);
    }

    int available() const { return (int)free_.size() + (int)evictable_.size(); }
    int cached() const { return (int)evictable_.size(); }

    int add_sequence(int64_t id, const int32_t *tokens, int n, int *num_cached) {
        if (seqs_.count(id)) return pkv::fail(PKV_ERR_INVALID, "bm_add_sequence: sequence %lld exists", (long long)id);
        if (n < 0 || (n > 0 && !tokens)) return pkv::fail(PKV_ERR_INVALID, "bm_add_sequence: bad tokens");
        const int nblk = (n + kBs - 1) / kBs;
        if (nblk > max_blocks_) return pkv::fail(PKV_ERR_INVALID, "bm_add_sequence: %d tokens exceed the table", n);
        // leading full blocks found in the prefix index
        // A hit needs the same 16 token ids and, as its predecessor, the block
        // already matched (the same physical block, not handed out again
        // since): the whole prefix up to the block is then compared, and a
        // collision of the 64-bit chain hash cannot reuse the wrong KV.
        std::vector<int32_t> hits;
        uint64_t h = 0;
        int32_t prev = -1;
        for (int b = 0; prefix_ && (b + 1) * kBs <= n; b++) {
            const uint64_t hb = block_hash(h, tokens + b * kBs);
            auto it = index_.find(hb);
            if (it == index_.end()) break;
            const Block &cand = blocks_[it->second];
            if (memcmp(cand.tok.data(), tokens + b * kBs, sizeof(int32_t) * kBs) || cand.parent != prev ||
                (prev >= 0 && cand.parent_gen != blocks_[prev].gen))
                break;
            hits.push_back(it->second);
            h = hb;
            prev = it->second;
        }
        // hit blocks that are cached (unreferenced) leave the evictable set, so
        // they are not counted as available for the new blocks
        int hit_evictable = 0;
        for (int32_t b : hits) hit_evictable += blocks_[b].ref == 0;
        const int need = nblk - (int)hits.size();
        if (need > available() - hit_evictable)
            return pkv::fail(PKV_ERR_OOB, "bm_add_sequence: %d blocks needed, %d available", need,
                             available() - hit_evictable);
        Seq s;
        for (int32_t b : hits) take_ref(b);
        s.blocks = hits;
        s.len = (int)hits.size() * kBs;
        s.tail_hash = h;
        if (num_cached) *num_cached = s.len;
        // new blocks for the rest of the prompt
        while (s.len < n) {
            const int32_t b = allocate();
            Block &blk = blocks_[b];
            blk.ref = 1;
            blk.ntok = 0;
            s.blocks.push_back(b);
            while (blk.ntok < kBs && s.len < n) blk.tok[blk.ntok++] = tokens[s.len++];
            if (blk.ntok == kBs) register_full(s, b);
        }
        seqs_.emplace(id, std::move(s));
        return PKV_OK;
    }

    int fork(int64_t parent, int64_t child) {
        auto it = seqs_.find(parent);
        if (it == seqs_.end()) return pkv::fail(PKV_ERR_INVALID, "bm_fork: unknown sequence %lld", (long long)parent);
        if (seqs_.count(child)) return pkv::fail(PKV_ERR_INVALID, "bm_fork: sequence %lld exists", (long long)child);
        Seq s = it->second;
        for (int32_t b : s.blocks) take_ref(b);
        seqs_.emplace(child, std::move(s));
        return PKV_OK;
    }

    int append_tokens(const int64_t *ids, int n, const int32_t *tokens, int64_t *slots, int64_t *pairs,
                      int *num_pairs) {
        if (n < 0 || (n > 0 && (!ids || !tokens || !slots || !pairs)) || !num_pairs)
            return pkv::fail(PKV_ERR_INVALID, "bm_append_tokens: bad arguments");
        // check everything first, so that a failing call changes nothing
        int need = 0;
        std::unordered_map<int64_t, int> seen;
        for (int i = 0; i < n; i++) {
            auto it = seqs_.find(ids[i]);
            if (it == seqs_.end())
                return pkv::fail(PKV_ERR_INVALID, "bm_append_tokens: unknown sequence %lld", (long long)ids[i]);
            if (seen[ids[i]]++)
                return pkv::fail(PKV_ERR_INVALID, "bm_append_tokens: sequence %lld listed twice", (long long)ids[i]);
            const Seq &s = it->second;
            if (s.len % kBs == 0) {
                if (s.len / kBs + 1 > max_blocks_)
                    return pkv::fail(PKV_ERR_INVALID, "bm_append_tokens: sequence %lld is at the table width",
                                     (long long)ids[i]);
                need++;
            } else if (blocks_[s.blocks.back()].ref > 1) {
                need++;
            }
        }
        if (need > available())
            return pkv::fail(PKV_ERR_OOB, "bm_append_tokens: %d blocks needed, %d available", need, available());
        int np = 0;
        for (int i = 0; i < n; i++) {
            Seq &s = seqs_[ids[i]];
            if (s.len % kBs == 0) {
                const int32_t b = allocate();
                blocks_[b].ref = 1;
                blocks_[b].ntok = 0;
                s.blocks.push_back(b);
            } else if (blocks_[s.blocks.back()].ref > 1) {
                // copy-on-write of the shared, partly filled last block
                const int32_t old = s.blocks.back();
                const int32_t b = allocate();
                blocks_[b].ref = 1;
                blocks_[b].ntok = blocks_[old].ntok;
                blocks_[b].tok = blocks_[old].tok;
                drop_ref(old);
                s.blocks.back() = b;
                pairs[2 * np] = old;
                pairs[2 * np + 1] = b;
                np++;
            }
            const int32_t b = s.blocks.back();
            Block &blk = blocks_[b];
            slots[i] = (int64_t)b * kBs + s.len % kBs;
            blk.tok[blk.ntok++] = tokens[i];
            s.len++;
            if (blk.ntok == kBs) register_full(s, b);
        }
        *num_pairs = np;
        return PKV_OK;
    }

    int slots(int64_t id, int first, int n, int64_t *out) {
        auto it = seqs_.find(id);
        if (it == seqs_.end()) return pkv::fail(PKV_ERR_INVALID, "bm_slots: unknown sequence %lld", (long long)id);
        const Seq &s = it->second;
        if (first < 0 || n < 0 || first + n > s.len || (n > 0 && !out))
            return pkv::fail(PKV_ERR_INVALID, "bm_slots: tokens [%d, %d) outside the sequence", first, first + n);
        for (int i = 0; i < n; i++) {
            const int t = first + i;
            out[i] = (int64_t)s.blocks[t / kBs] * kBs + t % kBs;
        }
        return PKV_OK;
    }

    int free_sequence(int64_t id) {
        auto it = seqs_.find(id);
        if (it == seqs_.end()) return pkv::fail(PKV_ERR_INVALID, "bm_free_sequence: unknown sequence %lld", (long long)id);
        for (int32_t b : it->second.blocks) drop_ref(b);
        seqs_.erase(it);
        return PKV_OK;
    }

    int tables(const int64_t *ids, int n, int32_t *out, int width, int32_t *lens) {
        if (n < 0 || width <= 0 || (n > 0 && (!ids || !out)))
            return pkv::fail(PKV_ERR_INVALID, "bm_block_tables: bad arguments");
        for (int i = 0; i < n; i++) {
            auto it = seqs_.find(ids[i]);
            if (it == seqs_.end())
                return pkv::fail(PKV_ERR_INVALID, "bm_block_tables: unknown sequence %lld", (long long)ids[i]);
            if ((int)it->second.blocks.size() > width)
                return pkv::fail(PKV_ERR_INVALID, "bm_block_tables: %zu blocks exceed the width %d",
                                 it->second.blocks.size(), width);
        }
        for (int i = 0; i < n; i++) {
            const Seq &s = seqs_[ids[i]];
            int32_t *row = out + (size_t)i * width;
            for (int j = 0; j < width; j++) row[j] = j < (int)s.blocks.size() ? s.blocks[j] : -1;
            if (lens) lens[i] = s.len;
        }
        return PKV_OK;
    }

  private:
    // A block for new content: a free one, else the least recently used
    // cached one (dropped from the index).  The caller has checked that one
    // is available.
    int32_t allocate() {
        int32_t b;
        if (!free_.empty()) {
            b = free_.back();
            free_.pop_back();
        } else {
            auto it = evictable_.begin();
            b = it->second;
            evictable_.erase(it);
            unregister(b);
        }
        blocks_[b].last_use = ++clock_;
        blocks_[b].gen++;
        return b;
    }

    void take_ref(int32_t b) {
        Block &blk = blocks_[b];
        if (blk.ref == 0 && blk.registered) evictable_.erase({blk.last_use, b});
        blk.ref++;
        blk.last_use = ++clock_;
    }

    void drop_ref(int32_t b) {
        Block &blk = blocks_[b];
        if (--blk.ref > 0) return;
        if (blk.registered) {
            blk.last_use = ++clock_;
            evictable_.insert({blk.last_use, b});
        } else {
            blk.ntok = 0;
            free_.push_back(b);
        }
    }

    // b has just become full as the last block of s: extend the chain hash
    // and enter it in the index, with its predecessor, unless an identical
    // block is already there.
    void register_full(Seq &s, int32_t b) {
        Block &blk = blocks_[b];
        const uint64_t h = block_hash(s.tail_hash, blk.tok.data());
        s.tail_hash = h;
        if (!prefix_ || blk.registered || index_.count(h)) return;
        blk.registered = true;
        blk.hash = h;
        blk.parent = s.blocks.size() >= 2 ? s.blocks[s.blocks.size() - 2] : -1;
        blk.parent_gen = blk.parent >= 0 ? blocks_[blk.parent].gen : 0;
        index_[h] = b;
    }

    void unregister(int32_t b) {
        Block &blk = blocks_[b];
        if (!blk.registered) return;
        auto it = index_.find(blk.hash);
        if (it != index_.end() && it->second == b) index_.erase(it);
        blk.registered = false;
        blk.ntok = 0;
    }

    std::vector<Block> blocks_;
    std::vector<int32_t> free_;
    std::set<std::pair<uint64_t, int32_t>> evictable_;  // (last use, block), oldest first
    std::unordered_map<uint64_t, int32_t> index_;       // chain hash -> registered block
    std::unordered_map<int64_t, Seq> seqs_;
    uint64_t clock_ = 0;
    int max_blocks_;
    bool prefix_;
};

BlockManager *as_bm(void *p) { return static_cast<BlockManager *>(p); }

}  // namespace

extern "C" int pkv_bm_create(int num_blocks, int max_blocks_per_seq, int prefix_cache, void **bm) {
    if (!bm || num_blocks <= 0 || max_blocks_per_seq <= 0)
        return pkv::fail(PKV_ERR_INVALID, "bm_create: bad arguments");
    *bm = new BlockManager(num_blocks, max_blocks_per_seq, prefix_cache != 0);
    return PKV_OK;
}

extern "C" int pkv_bm_destroy(void *bm) {
    if (!bm) return pkv::fail(PKV_ERR_INVALID, "bm_destroy: null manager");
    delete as_bm(bm);
    return PKV_OK;
}

extern "C" int pkv_bm_num_free_blocks(void *bm, int *free_blocks, int *cached_blocks) {
    if (!bm || !free_blocks) return pkv::fail(PKV_ERR_INVALID, "bm_num_free_blocks: bad arguments");
    *free_blocks = as_bm(bm)->available();
    if (cached_blocks) *cached_blocks = as_bm(bm)->cached();
    return PKV_OK;
}

extern "C" int pkv_bm_add_sequence(void *bm, int64_t seq_id, const int32_t *tokens, int num_tokens,
                                   int *num_cached_tokens) {
    if (!bm) return pkv::fail(PKV_ERR_INVALID, "bm_add_sequence: null manager");
    return as_bm(bm)->add_sequence(seq_id, tokens, num_tokens, num_cached_tokens);
}

extern "C" int pkv_bm_fork(void *bm, int64_t parent, int64_t child) {
    if (!bm) return pkv::fail(PKV_ERR_INVALID, "bm_fork: null manager");
    return as_bm(bm)->fork(parent, child);
}

extern "C" int pkv_bm_append_tokens(void *bm, const int64_t *seq_ids, int n, const int32_t *tokens,
                                    int64_t *slot_mapping, int64_t *copy_pairs, int *num_pairs) {
    if (!bm) return pkv::fail(PKV_ERR_INVALID, "bm_append_tokens: null manager");
    return as_bm(bm)->append_tokens(seq_ids, n, tokens, slot_mapping, copy_pairs, num_pairs);
}

extern "C" int pkv_bm_slots(void *bm, int64_t seq_id, int first, int n, int64_t *slots) {
    if (!bm) return pkv::fail(PKV_ERR_INVALID, "bm_slots: null manager");
    return as_bm(bm)->slots(seq_id, first, n, slots);
}

extern "C" int pkv_bm_free_sequence(void *bm, int64_t seq_id) {
    if (!bm) return pkv::fail(PKV_ERR_INVALID, "bm_free_sequence: null manager");
    return as_bm(bm)->free_sequence(seq_id);
}

extern "C" int pkv_bm_block_tables(void *bm, const int64_t *seq_ids, int n, int32_t *tables, int max_blocks,
                                   int32_t *context_lens) {
    if (!bm) return pkv::fail(PKV_ERR_INVALID, "bm_block_tables: null manager");
    return as_bm(bm)->tables(seq_ids, n, tables, max_blocks, context_lens);
}
