// kv_pages.h -- host bookkeeping of a paged KV cache (plain C++, no CUDA).
//
// Continuous batching ("Inside nanochat Part 4: Understanding Inference", Continuous
// Batching) adds sequences to and removes them from a running batch; with a cache carved
// into fixed pages, a sequence holds only the pages its positions reach, a finished one
// returns them, and a cloned one (Batch Prefilling via Cache Replication) shares its
// source's pages instead of copying them.
//
// A page holds `rows` consecutive positions of one sequence, for every layer and kv head;
// page ids index a pool of `npages` pages.  table[s * pps + i] is the page of positions
// [i * rows, (i + 1) * rows) of sequence s (-1: none).  Pages are reference counted: a
// fork points the clones' tables at the source's pages; the first write into a page that
// more than one sequence holds gives the writer a copy first (copy on write).  Writes only
// ever append (positions >= the sequence's length), so the one page that can be both
// shared and written is the partly filled page holding position `len`.
//
// Every change the device must see is queued: table entries (updates) and page copies
// (copies: rows [0, rows) of page src into page dst); the caller launches them, in
// stream order, before the kernels that read the cache.
//
// Without paging (`contiguous`) sequence s owns page s of max_seq rows for good: nothing
// is allocated or freed, and a fork copies the source's rows into the clone's own page.
#pragma once

#include <vector>

namespace slm {

struct KvPages {
    struct Copy {
        int src, dst, rows;
    };
    bool contiguous = true;
    int B = 0, pps = 0, rows = 0, shift = 31, npages = 0;
    std::vector<int> table;      // [B][pps]
    std::vector<int> refc;       // [npages]
    std::vector<int> free_list;  // pages with refc 0, taken from the back
    std::vector<int> upd_idx, upd_val;  // queued table writes
    std::vector<Copy> copies;           // queued page copies

    // One page of max_seq rows per sequence (the plain layout).
    void init_contiguous(int max_batch, int max_seq) {
        contiguous = true;
        B = max_batch;
        pps = 1;
        rows = max_seq;
        shift = 31;
        npages = max_batch;
        table.assign(B, 0);
        refc.assign(npages, 1);
        free_list.clear();
        for (int s = 0; s < B; s++) {
            table[s] = s;
            upd_idx.push_back(s);
            upd_val.push_back(s);
        }
    }

    // Pages of `page_rows` (a power of two) positions, `pool` pages in all.
    void init_paged(int max_batch, int max_seq, int page_rows, int pool) {
        contiguous = false;
        B = max_batch;
        rows = page_rows;
        shift = 0;
        while ((1 << shift) < page_rows) shift++;
        pps = (max_seq + page_rows - 1) / page_rows;
        npages = pool;
        table.assign((size_t)B * pps, -1);
        refc.assign(npages, 0);
        free_list.clear();
        for (int p = npages - 1; p >= 0; p--) free_list.push_back(p);  // page 0 is taken first
    }

    int pages_free() const { return (int)free_list.size(); }

    // Pages sequence s still lacks to hold positions [0, to) (plus one for a copy on
    // write when it appends from `len` into a shared page).
    int pages_needed(int s, int len, int to) const {
        if (contiguous) return 0;
        int need = 0;
        const int last = (to + rows - 1) / rows;
        for (int i = 0; i < last; i++)
            if (table[(size_t)s * pps + i] < 0) need++;
        if (to > len && (len & (rows - 1)) != 0) {
            const int pg = table[(size_t)s * pps + (len >> shift)];
            if (pg >= 0 && refc[pg] > 1) need++;
        }
        return need;
    }

    // Make positions [len, to) of sequence s writable: every page of [0, to) allocated,
    // the page holding `len` private.  Check pages_needed against pages_free first: this
    // call assumes they suffice.
    void prepare(int s, int len, int to) {
        if (contiguous || to <= len) return;
        if ((len & (rows - 1)) != 0) {
            const size_t e = (size_t)s * pps + (len >> shift);
            const int pg = table[e];
            if (pg >= 0 && refc[pg] > 1) {
                const int fresh = take();
                copies.push_back({pg, fresh, len & (rows - 1)});
                refc[pg]--;
                set(e, fresh);
            }
        }
        const int last = (to + rows - 1) / rows;
        for (int i = 0; i < last; i++) {
            const size_t e = (size_t)s * pps + i;
            if (table[e] < 0) set(e, take());
        }
    }

    // Sequence s forgets its positions: its pages go back to the pool when no other
    // sequence holds them.
    void release(int s) {
        if (contiguous) return;
        for (int i = 0; i < pps; i++) {
            const size_t e = (size_t)s * pps + i;
            const int pg = table[e];
            if (pg < 0) continue;
            if (--refc[pg] == 0) free_list.push_back(pg);
            table[e] = -1;  // the device never reads an entry past a sequence's length
        }
    }

    // Sequence dst (empty) becomes a copy of positions [0, len) of sequence src.
    void fork(int src, int dst, int len) {
        if (contiguous) {
            copies.push_back({src, dst, len});
            return;
        }
        const int last = (len + rows - 1) / rows;
        for (int i = 0; i < last; i++) {
            const int pg = table[(size_t)src * pps + i];
            refc[pg]++;
            set((size_t)dst * pps + i, pg);
        }
    }

    void clear_queue() {
        upd_idx.clear();
        upd_val.clear();
        copies.clear();
    }

  private:
    int take() {
        const int pg = free_list.back();
        free_list.pop_back();
        refc[pg] = 1;
        return pg;
    }
    void set(size_t e, int pg) {
        table[e] = pg;
        upd_idx.push_back((int)e);
        upd_val.push_back(pg);
    }
};

}  // namespace slm
