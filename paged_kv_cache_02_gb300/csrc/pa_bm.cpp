// pa_bm.cpp -- host KV block manager: physical block allocator, reference counts,
// fork / append / free, the copy-on-write decision and swapping to a host pool
// (host memory only).
//
// What it follows: the vLLM post (devpress), "1. overall architecture" (a request
// is a list of logical blocks filled left to right; the block table maps them to
// physical blocks of a pre-cut pool and records how full the last one is; a new
// physical block is taken only when the last logical block is full; a finished
// request's blocks are freed), "2.1 parallel sampling" (physical blocks carry
// reference counts; a request about to write into a block whose count is above one
// gets a newly taken block into which the shared block is copied, and the shared
// count drops by one, so the last holder writes in place) and "3. scheduling and
// preemption" (eviction moves all of a request's blocks to CPU memory, managed by a
// CPU block allocator, and copies them back when it resumes); the vLLM-SOSP23 note,
// "core method" (fork / append / free as the primitives of sampling, beam search and
// shared prefixes). Pensieve's sub-requests are forks whose rows list the same
// blocks.
//
// How: sequences live in a slot vector indexed through a hash map of caller ids;
// each pool (device, host) is a ring buffer handing blocks out first in, first out
// (freed blocks join its back in table order) with a count per block; a step's
// appends are checked for space first (counting the copies that the order of the
// step implies), then applied, so an exhausted pool changes nothing; a swap maps each
// distinct block of the listed requests to one block of the other pool, so blocks
// they share stay shared. Every operation costs O(its tokens + blocks).
#include <stdint.h>
#include <string.h>

#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pa.h"

namespace {

struct Pool {
  int32_t size = 0;
  std::vector<int32_t> ref;            // reference count of each block
  std::vector<int32_t> ring;           // free blocks, FIFO over [head, head + n_free)
  int32_t head = 0, n_free = 0;
  std::vector<uint64_t> stamp;         // per-block scratch of one operation
  std::vector<int32_t> scratch;

  // `order`: every id once (NULL: 0, 1, 2, ...). False on a bad order.
  bool init(int32_t n, const int32_t* order) {
    size = n;
    ref.assign(n, 0);
    ring.resize(n);
    stamp.assign(n, 0);
    scratch.assign(n, 0);
    if (order) {
      std::vector<uint8_t> seen(n, 0);
      for (int32_t i = 0; i < n; ++i) {
        const int32_t b = order[i];
        if (b < 0 || b >= n || seen[b]) return false;
        seen[b] = 1;
        ring[i] = b;
      }
    } else {
      for (int32_t i = 0; i < n; ++i) ring[i] = i;
    }
    head = 0;
    n_free = n;
    return true;
  }
  int32_t take() {                     // the caller sets the count
    const int32_t b = ring[head];
    head = head + 1 == size ? 0 : head + 1;
    --n_free;
    return b;
  }
  void give(int32_t b) {
    int64_t tail = (int64_t)head + n_free;
    if (tail >= size) tail -= size;
    ring[tail] = b;
    ++n_free;
  }
  void unref(int32_t b) {
    if (--ref[b] == 0) give(b);
  }
};

}  // namespace

struct pa_bm_s {
  int32_t block_size = 0;
  Pool dev, host;
  struct Seq {
    std::vector<int32_t> table;        // block of each logical block (host pool if on_host)
    int64_t len = 0;                   // tokens held (#filled follows from it)
    uint64_t stamp = 0;                // operation that last listed it (duplicate check)
    bool on_host = false;
  };
  std::vector<Seq> seqs;
  std::vector<int32_t> spare;          // reusable indices into seqs
  std::unordered_map<int64_t, int32_t> index;
  uint64_t step = 0;

  Seq* find(int64_t id) {
    auto it = index.find(id);
    return it == index.end() ? nullptr : &seqs[it->second];
  }
  int32_t new_seq(int64_t id) {
    int32_t i;
    if (!spare.empty()) {
      i = spare.back();
      spare.pop_back();
    } else {
      i = (int32_t)seqs.size();
      seqs.emplace_back();
    }
    Seq& s = seqs[i];
    s.table.clear();
    s.len = 0;
    s.on_host = false;
    index.emplace(id, i);
    return i;
  }
};

extern "C" {

pa_status pa_bm_create(int32_t num_blocks, int32_t block_size, const int32_t* h_free_order,
                       pa_bm_t* out) {
  if (!out || num_blocks <= 0 || block_size <= 0) return PA_ERR_INVALID_ARG;
  *out = nullptr;
  pa_bm_s* bm = new (std::nothrow) pa_bm_s();
  if (!bm) return PA_ERR_INVALID_ARG;
  try {
    bm->block_size = block_size;
    if (!bm->dev.init(num_blocks, h_free_order)) {
      delete bm;
      return PA_ERR_INVALID_ARG;
    }
  } catch (...) {
    delete bm;
    return PA_ERR_INVALID_ARG;
  }
  *out = bm;
  return PA_OK;
}

pa_status pa_bm_set_host_pool(pa_bm_t bm, int32_t num_host_blocks,
                              const int32_t* h_free_order) {
  if (!bm || num_host_blocks <= 0 || bm->host.size != 0) return PA_ERR_INVALID_ARG;
  try {
    if (!bm->host.init(num_host_blocks, h_free_order)) {
      bm->host = Pool();
      return PA_ERR_INVALID_ARG;
    }
  } catch (...) {
    bm->host = Pool();
    return PA_ERR_INVALID_ARG;
  }
  return PA_OK;
}

pa_status pa_bm_destroy(pa_bm_t bm) {
  delete bm;
  return PA_OK;
}

pa_status pa_bm_add(pa_bm_t bm, int64_t seq) {
  if (!bm) return PA_ERR_INVALID_ARG;
  if (bm->index.count(seq)) return PA_ERR_INVALID_ARG;
  try {
    bm->new_seq(seq);
  } catch (...) {
    return PA_ERR_INVALID_ARG;
  }
  return PA_OK;
}

pa_status pa_bm_fork(pa_bm_t bm, int64_t parent, int64_t child) {
  if (!bm) return PA_ERR_INVALID_ARG;
  auto it = bm->index.find(parent);
  if (it == bm->index.end() || bm->index.count(child)) return PA_ERR_INVALID_ARG;
  const int32_t pi = it->second;
  if (bm->seqs[pi].on_host) return PA_ERR_INVALID_ARG;
  try {
    const int32_t ci = bm->new_seq(child);       // may grow seqs: index, not pointer
    bm->seqs[ci].table = bm->seqs[pi].table;
    bm->seqs[ci].len = bm->seqs[pi].len;
  } catch (...) {
    return PA_ERR_INVALID_ARG;
  }
  for (int32_t b : bm->seqs[pi].table) bm->dev.ref[b] += 1;
  return PA_OK;
}

pa_status pa_bm_free(pa_bm_t bm, int64_t seq) {
  if (!bm) return PA_ERR_INVALID_ARG;
  auto it = bm->index.find(seq);
  if (it == bm->index.end()) return PA_ERR_INVALID_ARG;
  pa_bm_s::Seq& s = bm->seqs[it->second];
  Pool& pool = s.on_host ? bm->host : bm->dev;
  for (int32_t b : s.table) pool.unref(b);
  s.table.clear();
  s.len = 0;
  s.on_host = false;
  bm->spare.push_back(it->second);
  bm->index.erase(it);
  return PA_OK;
}

pa_status pa_bm_append(pa_bm_t bm, const int64_t* h_seqs, const int32_t* h_counts,
                       int32_t n_seqs, int64_t* h_slots, int32_t* h_cow_src,
                       int32_t* h_cow_dst, int32_t* n_cow) {
  if (!bm || n_seqs < 0 || !n_cow) return PA_ERR_INVALID_ARG;
  *n_cow = 0;
  if (n_seqs == 0) return PA_OK;
  if (!h_seqs || !h_counts || !h_cow_src || !h_cow_dst) return PA_ERR_INVALID_ARG;
  const int64_t B = bm->block_size;
  Pool& dev = bm->dev;
  const uint64_t step = ++bm->step;
  // ---- check: known, on the device, listed once, counts >= 0; free blocks needed
  int64_t need = 0, total = 0;
  std::vector<int32_t> idx(n_seqs);
  for (int32_t i = 0; i < n_seqs; ++i) {
    auto it = bm->index.find(h_seqs[i]);
    if (it == bm->index.end() || h_counts[i] < 0) return PA_ERR_INVALID_ARG;
    pa_bm_s::Seq& s = bm->seqs[it->second];
    if (s.on_host || s.stamp == step) return PA_ERR_INVALID_ARG;
    s.stamp = step;
    idx[i] = it->second;
    const int64_t n = h_counts[i];
    if (n == 0) continue;
    total += n;
    if (s.len % B != 0) {
      const int32_t last = s.table.back();
      if (dev.stamp[last] != step) {     // counts left after earlier copies of the step
        dev.stamp[last] = step;
        dev.scratch[last] = dev.ref[last];
      }
      if (dev.scratch[last] > 1) {       // this writer copies; the count drops by one
        need += 1;
        dev.scratch[last] -= 1;
      }
    }
    need += (s.len + n + B - 1) / B - (int64_t)s.table.size();
  }
  if (total > 0 && !h_slots) return PA_ERR_INVALID_ARG;
  if (need > dev.n_free) return PA_ERR_NO_SPACE;
  // ---- apply, in the listed order
  int64_t k = 0;
  int32_t nc = 0;
  for (int32_t i = 0; i < n_seqs; ++i) {
    pa_bm_s::Seq& s = bm->seqs[idx[i]];
    const int64_t n = h_counts[i];
    for (int64_t p = s.len; p < s.len + n; ++p) {
      const int64_t j = p / B;
      if (j == (int64_t)s.table.size()) {
        const int32_t b = dev.take();
        dev.ref[b] = 1;
        s.table.push_back(b);
      } else if (dev.ref[s.table[j]] > 1) {
        const int32_t old = s.table[j];
        const int32_t fresh = dev.take();
        dev.ref[fresh] = 1;
        dev.ref[old] -= 1;
        h_cow_src[nc] = old;
        h_cow_dst[nc] = fresh;
        ++nc;
        s.table[j] = fresh;
      }
      h_slots[k++] = (int64_t)s.table[j] * B + p % B;
    }
    s.len += n;
  }
  *n_cow = nc;
  return PA_OK;
}

// Swap of the listed requests from pool `from` to pool `to` (out: device -> host).
static pa_status bm_swap(pa_bm_t bm, const int64_t* h_seqs, int32_t n_seqs, bool out,
                         int32_t* h_from, int32_t* h_to, int32_t capacity, int32_t* n_pairs) {
  if (!bm || n_seqs < 0 || capacity < 0 || !n_pairs) return PA_ERR_INVALID_ARG;
  *n_pairs = 0;
  if (n_seqs == 0) return PA_OK;
  if (!h_seqs) return PA_ERR_INVALID_ARG;
  Pool& from = out ? bm->dev : bm->host;
  Pool& to = out ? bm->host : bm->dev;
  const uint64_t step = ++bm->step;
  // ---- check: known, listed once, on the side they leave; distinct blocks
  std::vector<int32_t> idx(n_seqs);
  int64_t distinct = 0;
  for (int32_t i = 0; i < n_seqs; ++i) {
    auto it = bm->index.find(h_seqs[i]);
    if (it == bm->index.end()) return PA_ERR_INVALID_ARG;
    pa_bm_s::Seq& s = bm->seqs[it->second];
    if (s.on_host != !out || s.stamp == step) return PA_ERR_INVALID_ARG;
    s.stamp = step;
    idx[i] = it->second;
    for (int32_t b : s.table)
      if (from.stamp[b] != step) {
        from.stamp[b] = step;
        ++distinct;
      }
  }
  if (distinct > to.n_free) return PA_ERR_NO_SPACE;
  if (distinct > capacity || (distinct > 0 && (!h_from || !h_to))) return PA_ERR_SHAPE;
  // ---- apply: one block of `to` per distinct block, in the order the tables name them
  const uint64_t apply = ++bm->step;
  int32_t np = 0;
  for (int32_t i = 0; i < n_seqs; ++i)
    for (int32_t b : bm->seqs[idx[i]].table)
      if (from.stamp[b] != apply) {
        from.stamp[b] = apply;
        const int32_t c = to.take();
        to.ref[c] = 0;
        from.scratch[b] = c;
        h_from[np] = b;
        h_to[np] = c;
        ++np;
      }
  for (int32_t i = 0; i < n_seqs; ++i) {
    pa_bm_s::Seq& s = bm->seqs[idx[i]];
    for (int32_t& b : s.table) {
      const int32_t c = from.scratch[b];
      to.ref[c] += 1;
      from.unref(b);
      b = c;
    }
    s.on_host = out;
  }
  *n_pairs = np;
  return PA_OK;
}

pa_status pa_bm_swap_out(pa_bm_t bm, const int64_t* h_seqs, int32_t n_seqs, int32_t* h_dev,
                         int32_t* h_host, int32_t capacity, int32_t* n_pairs) {
  return bm_swap(bm, h_seqs, n_seqs, true, h_dev, h_host, capacity, n_pairs);
}

pa_status pa_bm_swap_in(pa_bm_t bm, const int64_t* h_seqs, int32_t n_seqs, int32_t* h_host,
                        int32_t* h_dev, int32_t capacity, int32_t* n_pairs) {
  return bm_swap(bm, h_seqs, n_seqs, false, h_host, h_dev, capacity, n_pairs);
}

pa_status pa_bm_tables(pa_bm_t bm, const int64_t* h_seqs, int32_t n_seqs, int32_t max_blocks,
                       int32_t* h_block_table, int32_t* h_context_lens) {
  if (!bm || n_seqs < 0 || max_blocks < 0) return PA_ERR_INVALID_ARG;
  if (n_seqs == 0) return PA_OK;
  if (!h_seqs || (!h_block_table && !h_context_lens)) return PA_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n_seqs; ++i) {
    const pa_bm_s::Seq* s = bm->find(h_seqs[i]);
    if (!s) return PA_ERR_INVALID_ARG;
    if (h_block_table && (int64_t)s->table.size() > max_blocks) return PA_ERR_SHAPE;
    if (h_context_lens && s->len > INT32_MAX) return PA_ERR_RANGE;
  }
  for (int32_t i = 0; i < n_seqs; ++i) {
    const pa_bm_s::Seq* s = bm->find(h_seqs[i]);
    if (h_block_table) {
      int32_t* row = h_block_table + (int64_t)i * max_blocks;
      const int32_t nb = (int32_t)s->table.size();
      if (nb) memcpy(row, s->table.data(), sizeof(int32_t) * nb);
      for (int32_t j = nb; j < max_blocks; ++j) row[j] = -1;
    }
    if (h_context_lens) h_context_lens[i] = (int32_t)s->len;
  }
  return PA_OK;
}

pa_status pa_bm_seq_info(pa_bm_t bm, int64_t seq, int64_t* len, int32_t* n_blocks,
                         int32_t* on_host) {
  if (!bm) return PA_ERR_INVALID_ARG;
  const pa_bm_s::Seq* s = bm->find(seq);
  if (!s) return PA_ERR_INVALID_ARG;
  if (len) *len = s->len;
  if (n_blocks) *n_blocks = (int32_t)s->table.size();
  if (on_host) *on_host = s->on_host ? 1 : 0;
  return PA_OK;
}

pa_status pa_bm_refcount(pa_bm_t bm, int32_t block, int32_t* count) {
  if (!bm || !count) return PA_ERR_INVALID_ARG;
  if (block < 0 || block >= bm->dev.size) return PA_ERR_RANGE;
  *count = bm->dev.ref[block];
  return PA_OK;
}

pa_status pa_bm_host_refcount(pa_bm_t bm, int32_t block, int32_t* count) {
  if (!bm || !count) return PA_ERR_INVALID_ARG;
  if (block < 0 || block >= bm->host.size) return PA_ERR_RANGE;
  *count = bm->host.ref[block];
  return PA_OK;
}

pa_status pa_bm_num_free(pa_bm_t bm, int32_t* n_free) {
  if (!bm || !n_free) return PA_ERR_INVALID_ARG;
  *n_free = bm->dev.n_free;
  return PA_OK;
}

pa_status pa_bm_host_num_free(pa_bm_t bm, int32_t* n_free) {
  if (!bm || !n_free) return PA_ERR_INVALID_ARG;
  *n_free = bm->host.n_free;
  return PA_OK;
}

}  // extern "C"
