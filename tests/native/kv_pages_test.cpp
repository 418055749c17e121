// Host test of the paged KV cache bookkeeping (kv_pages.h), built and run by
// tests/test_kv_pages.py with the system C++ compiler.  A simulated device memory
// (every page a row of ints) receives the queued page copies and each step's writes;
// every sequence must always read back exactly what was written at its own positions
// (directly, or before a fork by the sequence it was cloned from).  Prints "ok" or the
// first failure and exits nonzero.
#include <cstdio>
#include <cstdlib>
#include <map>
#include <vector>

#include "kv_pages.h"

using slm::KvPages;

static int fails = 0;
#define CHECK(cond, ...)                                   \
    do {                                                   \
        if (!(cond)) {                                     \
            std::printf("FAIL line %d: ", __LINE__);       \
            std::printf(__VA_ARGS__);                      \
            std::printf("\n");                             \
            if (++fails > 5) std::exit(1);                 \
        }                                                  \
    } while (0)

struct Sim {
    KvPages kp;
    std::vector<std::vector<long>> mem;     // [page][row]
    std::vector<int> dtable;                // the device's copy of the table
    std::vector<std::vector<long>> expect;  // [seq][pos] value the sequence must read
    std::vector<int> len;
    long next_value = 1;

    void init(int B, int max_seq, int rows, int pool) {
        kp.init_paged(B, max_seq, rows, pool);
        mem.assign(pool, std::vector<long>(rows, 0));
        dtable.assign(kp.table.size(), -1);
        expect.assign(B, {});
        len.assign(B, 0);
    }
    void flush() {  // what the library launches, in the same order
        for (auto &c : kp.copies)
            for (int r = 0; r < c.rows; r++) mem[c.dst][r] = mem[c.src][r];
        for (size_t i = 0; i < kp.upd_idx.size(); i++) dtable[kp.upd_idx[i]] = kp.upd_val[i];
        kp.clear_queue();
    }
    long &cell(int s, int p) {
        const int pg = dtable[(size_t)s * kp.pps + (p >> kp.shift)];
        CHECK(pg >= 0 && pg < kp.npages, "seq %d pos %d: no page on the device", s, p);
        return mem[pg < 0 ? 0 : pg][p & (kp.rows - 1)];
    }
    // append n positions to sequence s (what a prefill or decode steps write)
    bool append(int s, int n) {
        if (kp.pages_needed(s, len[s], len[s] + n) > kp.pages_free()) return false;
        kp.prepare(s, len[s], len[s] + n);
        flush();
        for (int i = 0; i < n; i++) {
            const long v = next_value++;
            cell(s, len[s] + i) = v;
            expect[s].push_back(v);
        }
        len[s] += n;
        return true;
    }
    void fork(int src, int dst) {
        kp.fork(src, dst, len[src]);
        flush();
        expect[dst] = expect[src];
        len[dst] = len[src];
    }
    void reset(int s) {
        kp.release(s);
        expect[s].clear();
        len[s] = 0;
    }
    void verify() {
        for (int s = 0; s < (int)len.size(); s++)
            for (int p = 0; p < len[s]; p++)
                CHECK(cell(s, p) == expect[s][p], "seq %d pos %d reads %ld, wrote %ld", s, p, cell(s, p), expect[s][p]);
        // reference counts equal the number of table entries that hold each page
        std::vector<int> held(kp.npages, 0);
        for (int e : kp.table)
            if (e >= 0) held[e]++;
        int free_count = 0;
        for (int p = 0; p < kp.npages; p++) {
            CHECK(held[p] == kp.refc[p], "page %d held %d times, refc %d", p, held[p], kp.refc[p]);
            if (held[p] == 0) free_count++;
        }
        CHECK(free_count == kp.pages_free(), "free list %d, unheld pages %d", kp.pages_free(), free_count);
    }
};

int main() {
    {  // walk-through: 16-row pages, fork in mid-page, copy on write, release
        Sim m;
        m.init(4, 128, 16, 20);
        CHECK(m.append(0, 40), "append");
        CHECK(m.kp.pages_free() == 17, "3 pages for 40 positions, free %d", m.kp.pages_free());
        m.fork(0, 1);
        CHECK(m.kp.pages_free() == 17, "a fork takes no page, free %d", m.kp.pages_free());
        for (int i = 0; i < 3; i++) CHECK(m.kp.table[m.kp.pps + i] == m.kp.table[i], "clone shares page %d", i);
        CHECK(m.kp.pages_needed(1, 40, 41) == 1, "the shared partial page needs a copy");
        CHECK(m.append(1, 1), "append to the clone");
        CHECK(m.kp.pages_free() == 16, "copy on write took one page, free %d", m.kp.pages_free());
        CHECK(m.kp.table[m.kp.pps + 2] != m.kp.table[2], "the clone's third page is private");
        CHECK(m.kp.table[m.kp.pps + 1] == m.kp.table[1], "full pages stay shared");
        CHECK(m.kp.pages_needed(0, 40, 41) == 0, "the source's page is private again");
        CHECK(m.append(0, 1), "append to the source");
        CHECK(m.kp.pages_free() == 16, "no copy for the source, free %d", m.kp.pages_free());
        m.verify();
        m.reset(0);
        CHECK(m.kp.pages_free() == 17, "only the source's private page returns, free %d", m.kp.pages_free());
        m.verify();
        m.reset(1);
        CHECK(m.kp.pages_free() == 20, "every page returns, free %d", m.kp.pages_free());
        m.fork(2, 3);  // forking an empty sequence shares nothing
        CHECK(m.kp.pages_free() == 20, "empty fork");
    }
    {  // a fork at a page boundary copies nothing on the next write
        Sim m;
        m.init(2, 64, 16, 8);
        CHECK(m.append(0, 32), "append");
        m.fork(0, 1);
        CHECK(m.kp.pages_needed(1, 32, 33) == 1, "one new page, no copy");
        CHECK(m.append(1, 1), "append");
        CHECK(m.kp.copies.empty(), "queue flushed");
        m.verify();
    }
    {  // exhaustion: nothing changes, then room after a reset
        Sim m;
        m.init(2, 64, 16, 4);
        CHECK(m.append(0, 48), "append");
        CHECK(!m.append(1, 17), "two pages needed, one free");
        CHECK(m.kp.pages_free() == 1 && m.len[1] == 0, "a refused append takes nothing");
        CHECK(m.append(1, 16), "one page");
        CHECK(!m.append(0, 1), "the pool is empty");
        m.reset(1);
        CHECK(m.append(0, 1), "room after the reset");
        m.verify();
    }
    {  // random walks: appends, forks, resets on 6 slots of a 40-page pool
        for (int seed = 1; seed <= 40; seed++) {
            std::srand(seed);
            Sim m;
            const int rows = seed % 2 ? 16 : 32;
            m.init(6, 256, rows, 40);
            for (int op = 0; op < 400; op++) {
                const int s = std::rand() % 6, r = std::rand() % 10;
                if (r < 6) {
                    const int n = 1 + (r == 0 ? std::rand() % 70 : 0);
                    if (m.len[s] + n <= 256) m.append(s, n);
                } else if (r < 8) {
                    int d = std::rand() % 6;
                    if (d != s && m.len[d] == 0 && m.len[s] > 0) m.fork(s, d);
                } else {
                    m.reset(s);
                }
                if (op % 25 == 0) m.verify();
            }
            m.verify();
        }
    }
    if (fails) return 1;
    std::printf("ok\n");
    return 0;
}
