// Host-side block manager with a prefix cache: the bookkeeping half of
// PagedAttention, native, behind the library's C ABI.
//
// Model (CS349E Lecture 7 notes §4.1, §5.1, §8; Month 2 · PagedAttention,
// infra learning path, §6.2-§7.5):
//   * the pool is num_blocks physical blocks of block_size tokens; a sequence
//     owns a list of block ids (its block table) and gets a new block only
//     when its last one is full;
//   * fork shares every block (reference count + 1); appending into a shared,
//     partially filled last block first copies it (copy-on-write) and reports
//     the (src, dst) pair for pa_copy_blocks;
//   * with prefix caching on, every full block is identified by a chain hash
//     h_i = H(h_{i-1}, tokens of block i), so a hit means the whole prefix up
//     to and including that block matches; a new sequence reuses the cached
//     blocks of its longest matching block-aligned prefix;
//   * a block whose count drops to zero and that holds a cached full block is
//     kept, reusable, on an LRU list; a block is evicted (its hash forgotten)
//     only when no never-used or uncached free block is left, least recently
//     released first. Blocks of a freed sequence are released tail first, so
//     the shared head of a prefix is evicted last.
// Hash matches are confirmed against the stored parent hash and tokens, so a
// hash collision can never hand out the wrong block.
#include <cstdint>
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa.h"

namespace {

uint64_t mix64(uint64_t x) {  // SplitMix64 finaliser
  x += 0x9e3779b97f4a7c15ull;
  x = (x ^ (x >> 30)) * 0xbf58476d1ce4e5b9ull;
  x = (x ^ (x >> 27)) * 0x94d049bb133111ebull;
  return x ^ (x >> 31);
}

uint64_t chain_hash(uint64_t parent, const int32_t* tokens, int n) {
  uint64_t h = mix64(parent ^ 0x5851f42d4c957f2dull);
  for (int i = 0; i < n; ++i) h = mix64(h ^ static_cast<uint32_t>(tokens[i]));
  return h | 1ull;  // 0 means "no hash"
}

struct Block {
  int32_t ref = 0;
  uint64_t hash = 0;       // chain hash while the block is registered in the prefix cache
  uint64_t parent = 0;     // parent hash it was registered with
  std::vector<int32_t> tokens;
  int64_t prev = -1, next = -1;  // links in the free or LRU list
  int8_t list = 0;               // 0 none, 1 free, 2 LRU (evictable)
};

struct Seq {
  std::vector<int64_t> blocks;
  std::vector<int32_t> tokens;
  std::vector<uint64_t> hashes;  // chain hash of each full block (0 for blocks not hashed)
};

struct List {
  int64_t head = -1, tail = -1, size = 0;
};

}  // namespace

struct pa_bm {
  int64_t num_blocks;
  int block_size;
  bool caching;
  std::vector<Block> blocks;
  List free_list;  // never used or holding nothing reusable
  List lru;        // refcount 0, holding a cached full block; head = least recently released
  std::unordered_map<uint64_t, int64_t> cache;
  std::unordered_map<int64_t, Seq> seqs;
  int64_t queries = 0, hits = 0, evictions = 0, copies = 0;

  void push_back(List& l, int8_t tag, int64_t b) {
    Block& x = blocks[b];
    x.prev = l.tail;
    x.next = -1;
    x.list = tag;
    if (l.tail >= 0) blocks[l.tail].next = b; else l.head = b;
    l.tail = b;
    ++l.size;
  }
  void unlink(List& l, int64_t b) {
    Block& x = blocks[b];
    if (x.prev >= 0) blocks[x.prev].next = x.next; else l.head = x.next;
    if (x.next >= 0) blocks[x.next].prev = x.prev; else l.tail = x.prev;
    x.prev = x.next = -1;
    x.list = 0;
    --l.size;
  }
  void forget(int64_t b) {
    Block& x = blocks[b];
    if (x.hash) {
      auto it = cache.find(x.hash);
      if (it != cache.end() && it->second == b) cache.erase(it);
    }
    x.hash = x.parent = 0;
    x.tokens.clear();
  }
  // A block for new content: a free one, else evict the least recently released cached one.
  int64_t take() {
    int64_t b = -1;
    if (free_list.size) {
      b = free_list.head;
      unlink(free_list, b);
    } else if (lru.size) {
      b = lru.head;
      unlink(lru, b);
      forget(b);
      ++evictions;
    } else {
      return -1;
    }
    blocks[b].ref = 1;
    return b;
  }
  void release(int64_t b) {
    Block& x = blocks[b];
    if (--x.ref > 0) return;
    if (caching && x.hash) push_back(lru, 2, b); else { forget(b); push_back(free_list, 1, b); }
  }
  // Register full block i of sequence s in the prefix cache.
  void register_full(Seq& s, size_t i) {
    const int B = block_size;
    const uint64_t parent = (i && i - 1 < s.hashes.size()) ? s.hashes[i - 1] : 0;
    if (s.hashes.size() <= i) s.hashes.resize(i + 1, 0);
    if (!caching || (i && !parent)) return;
    const uint64_t h = chain_hash(parent, s.tokens.data() + i * B, B);
    s.hashes[i] = h;
    const int64_t b = s.blocks[i];
    Block& x = blocks[b];
    if (x.hash || cache.count(h)) return;  // already registered (shared block) or an equal block exists
    x.hash = h;
    x.parent = parent;
    x.tokens.assign(s.tokens.begin() + i * B, s.tokens.begin() + (i + 1) * B);
    cache.emplace(h, b);
  }
  // Cached block for full block i of a prompt with the given parent hash, or -1.
  int64_t lookup(uint64_t parent, const int32_t* toks) {
    const uint64_t h = chain_hash(parent, toks, block_size);
    auto it = cache.find(h);
    if (it == cache.end()) return -1;
    const Block& x = blocks[it->second];
    if (x.parent != parent || std::memcmp(x.tokens.data(), toks, sizeof(int32_t) * block_size) != 0) return -1;
    return it->second;
  }
};

extern "C" pa_bm* pa_bm_create(int64_t num_blocks, int block_size, int prefix_caching) {
  if (num_blocks <= 0 || block_size <= 0 || num_blocks > (1LL << 40)) return nullptr;
  pa_bm* m = new (std::nothrow) pa_bm();
  if (!m) return nullptr;
  m->num_blocks = num_blocks;
  m->block_size = block_size;
  m->caching = prefix_caching != 0;
  m->blocks.resize(num_blocks);
  for (int64_t b = 0; b < num_blocks; ++b) m->push_back(m->free_list, 1, b);
  return m;
}

extern "C" void pa_bm_destroy(pa_bm* m) { delete m; }

extern "C" pa_status pa_bm_add_sequence(pa_bm* m, int64_t seq_id, const int32_t* tokens, int32_t num_tokens,
                                        int32_t* cached_tokens) {
  if (!m || num_tokens < 0 || (num_tokens && !tokens) || m->seqs.count(seq_id)) return PA_ERR_INVALID_ARG;
  const int B = m->block_size;
  const int64_t nblk = (num_tokens + B - 1) / B, nfull = num_tokens / B;
  Seq s;
  s.tokens.assign(tokens, tokens + num_tokens);
  // longest cached block-aligned prefix
  std::vector<int64_t> hit;
  uint64_t parent = 0;
  if (m->caching) {
    for (int64_t i = 0; i < nfull; ++i) {
      ++m->queries;
      const int64_t b = m->lookup(parent, tokens + i * B);
      if (b < 0) break;
      hit.push_back(b);
      parent = m->blocks[b].hash;
    }
  }
  // blocks needed beyond the hits must be available (hits on evictable blocks also leave the pool)
  int64_t hit_evictable = 0;
  for (int64_t b : hit) hit_evictable += m->blocks[b].ref == 0;
  if (nblk - (int64_t)hit.size() > m->free_list.size + m->lru.size - hit_evictable) return PA_ERR_NO_BLOCKS;
  for (int64_t b : hit) {
    Block& x = m->blocks[b];
    if (x.ref == 0) m->unlink(m->lru, b);
    ++x.ref;
    s.blocks.push_back(b);
    s.hashes.push_back(x.hash);
  }
  m->hits += (int64_t)hit.size();
  for (int64_t i = (int64_t)hit.size(); i < nblk; ++i) s.blocks.push_back(m->take());
  for (int64_t i = (int64_t)hit.size(); i < nfull; ++i) m->register_full(s, (size_t)i);
  if (cached_tokens) *cached_tokens = (int32_t)(hit.size() * B);
  m->seqs.emplace(seq_id, std::move(s));
  return PA_OK;
}

extern "C" pa_status pa_bm_fork(pa_bm* m, int64_t parent, int64_t child) {
  if (!m || m->seqs.count(child)) return PA_ERR_INVALID_ARG;
  auto it = m->seqs.find(parent);
  if (it == m->seqs.end()) return PA_ERR_INVALID_ARG;
  Seq c = it->second;
  for (int64_t b : c.blocks) ++m->blocks[b].ref;
  m->seqs.emplace(child, std::move(c));
  return PA_OK;
}

extern "C" pa_status pa_bm_append(pa_bm* m, int64_t seq_id, int32_t token, int64_t* slot, int64_t* cow_src,
                                  int64_t* cow_dst) {
  if (!m) return PA_ERR_INVALID_ARG;
  auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end()) return PA_ERR_INVALID_ARG;
  Seq& s = it->second;
  const int B = m->block_size;
  const int64_t n = (int64_t)s.tokens.size();
  const int off = (int)(n % B);
  int64_t src = -1, dst = -1;
  if (off == 0) {
    const int64_t b = m->take();
    if (b < 0) return PA_ERR_NO_BLOCKS;
    s.blocks.push_back(b);
  } else {
    const int64_t last = s.blocks.back();
    if (m->blocks[last].ref > 1) {  // shared partial block: copy before writing
      const int64_t b = m->take();
      if (b < 0) return PA_ERR_NO_BLOCKS;
      --m->blocks[last].ref;
      s.blocks.back() = b;
      src = last;
      dst = b;
      ++m->copies;
    }
  }
  s.tokens.push_back(token);
  if (off == B - 1) m->register_full(s, s.blocks.size() - 1);
  if (slot) *slot = s.blocks.back() * B + off;
  if (cow_src) *cow_src = src;
  if (cow_dst) *cow_dst = dst;
  return PA_OK;
}

extern "C" pa_status pa_bm_free(pa_bm* m, int64_t seq_id) {
  if (!m) return PA_ERR_INVALID_ARG;
  auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end()) return PA_ERR_INVALID_ARG;
  const std::vector<int64_t>& bl = it->second.blocks;
  for (auto r = bl.rbegin(); r != bl.rend(); ++r) m->release(*r);  // tail first
  m->seqs.erase(it);
  return PA_OK;
}

extern "C" int32_t pa_bm_block_table(const pa_bm* m, int64_t seq_id, int32_t* out, int32_t capacity) {
  if (!m) return -1;
  auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end()) return -1;
  const std::vector<int64_t>& bl = it->second.blocks;
  const int32_t n = (int32_t)bl.size();
  for (int32_t i = 0; i < n && i < capacity; ++i) out[i] = (int32_t)bl[i];
  return n;
}

extern "C" int64_t pa_bm_context_len(const pa_bm* m, int64_t seq_id) {
  if (!m) return -1;
  auto it = m->seqs.find(seq_id);
  return it == m->seqs.end() ? -1 : (int64_t)it->second.tokens.size();
}

extern "C" int64_t pa_bm_num_free(const pa_bm* m) { return m ? m->free_list.size + m->lru.size : -1; }

extern "C" void pa_bm_stats(const pa_bm* m, int64_t* out) {
  if (!m || !out) return;
  out[0] = m->queries;
  out[1] = m->hits;
  out[2] = m->evictions;
  out[3] = m->copies;
  out[4] = m->lru.size;
  out[5] = (int64_t)m->cache.size();
}
