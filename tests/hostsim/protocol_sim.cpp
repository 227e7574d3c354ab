// Host-thread emulation of the publish / last-arriver protocol of the fused
// GEMV + one-shot all-reduce (TEST INFRASTRUCTURE: compiled and driven by
// tests/test_protocol_sim.py on the CPU; nothing in the library uses it).
//
// R threads play the R ranks.  A launch reads its epoch e from the epoch
// word (one more than the last finished launch).  Each rank, for every tile t
// of the launch in its own (shuffled) order, writes its partial of tile t and
// its flag flags[r][t] = e (relaxed), fences, and takes an arrival ticket
// with an acq_rel fetch_add on counters[t].  Tickets run 0..R-1 in every
// launch; the holder of R-1 counts the tile on tiles_done, puts the counter
// back to zero, reads the R flags (each must equal e; the acq_rel ticket
// orders these loads after every rank's fenced stores), sums the R partials
// in rank order 0..R-1 and writes y[t]; the reducer of the last tile stores e into the
// epoch word and clears tiles_done.  No thread waits for another; a ticket out of
// range or a stale flag latches a status code, and a rank made to skip a tile
// latches the code of a CTA that gave up (as the kernels' bounded waits do).
// This is the protocol of the fused GEMV + AllReduce ("Overlapping Collective
// Communication with Dependent Computation ...", Abstract: partials pushed as
// soon as each share is done, the reduction by whoever completes a tile) and
// the symmetric-memory one-shot all-reduce, played by threads instead of CTAs.
//
// The bounded wait of the multi-GPU design -- a reducer that waits for the R
// flags of its tile with a deadline and reports a timeout instead of hanging
// -- is emulated by sim_wait_flags.
#include <algorithm>
#include <atomic>
#include <chrono>
#include <cstdint>
#include <cstring>
#include <limits>
#include <random>
#include <thread>
#include <vector>

namespace {

struct Shared {
    int R, T;
    std::vector<std::atomic<uint32_t>> flags;     // [R][T]
    std::vector<std::atomic<uint32_t>> counters;  // [T]
    std::atomic<uint32_t> epoch_word{0};          // epoch of the last finished launch
    std::atomic<uint32_t> tiles_done{0};
    std::vector<double> partial;                  // [R][T] (plain: ordered by the fence and the acq_rel ticket)
    std::vector<double> y;                        // [T]
    std::atomic<int> status{0};
    std::atomic<int> bad_tile{-1};
    Shared(int R_, int T_) : R(R_), T(T_), flags((size_t)R_ * T_), counters((size_t)T_), partial((size_t)R_ * T_),
                             y((size_t)T_) {
        for (auto &f : flags) f.store(0);
        for (auto &c : counters) c.store(0);
    }
};

Shared *g = nullptr;

void latch(int code, int t) {
    int zero = 0;
    if (g->status.compare_exchange_strong(zero, code)) g->bad_tile.store(t);
}

// One rank's launch over tiles 0..tiles-1.  skip_tile >= 0: this rank gives
// up before publishing that tile (and latches code 3, as a CTA whose bounded
// wait ran out does); stale_tile >= 0: it publishes that tile with the
// previous epoch.
void rank_launch(int r, int tiles, const double *values, unsigned seed, int skip_tile, int stale_tile,
                 int max_sleep_us) {
    const uint32_t epoch = g->epoch_word.load(std::memory_order_relaxed) + 1u;
    std::vector<int> order((size_t)tiles);
    for (int t = 0; t < tiles; ++t) order[(size_t)t] = t;
    std::mt19937 rng(seed);
    std::shuffle(order.begin(), order.end(), rng);
    std::uniform_int_distribution<int> pause(0, max_sleep_us > 0 ? max_sleep_us : 0);
    const uint32_t C = (uint32_t)g->R;
    for (int t : order) {
        if (t == skip_tile) {
            latch(3, t);
            continue;
        }
        if (max_sleep_us > 0) std::this_thread::sleep_for(std::chrono::microseconds(pause(rng)));
        g->partial[(size_t)r * g->T + t] = values[(size_t)r * g->T + t];
        g->flags[(size_t)r * g->T + t].store(t == stale_tile ? epoch - 1 : epoch, std::memory_order_relaxed);
        std::atomic_thread_fence(std::memory_order_release);
        const uint32_t pos = g->counters[(size_t)t].fetch_add(1u, std::memory_order_acq_rel);
        if (pos >= C) {
            latch(2, t);   // bad ticket: launches overlapped or the pad was not reset
            continue;
        }
        if (pos != C - 1u) continue;
        // The reducer: count the tile, put the counter back to zero (every
        // contributor has arrived), check the flags, advance the epoch if
        // this was the launch's last tile, then reduce.
        const uint32_t done = g->tiles_done.fetch_add(1u, std::memory_order_release);
        g->counters[(size_t)t].store(0u, std::memory_order_relaxed);
        bool ok = true;
        for (int q = 0; q < g->R; ++q)
            if (g->flags[(size_t)q * g->T + t].load(std::memory_order_relaxed) != epoch) ok = false;
        if (done >= (uint32_t)tiles) latch(2, t);
        if (done == (uint32_t)tiles - 1u) {   // the last tile: every rank has read the epoch
            std::atomic_thread_fence(std::memory_order_acquire);
            g->tiles_done.store(0u, std::memory_order_relaxed);
            g->epoch_word.store(epoch, std::memory_order_relaxed);
        }
        if (!ok) {
            latch(1, t);   // stale or missing flag
            continue;
        }
        double acc = 0.0;
        for (int q = 0; q < g->R; ++q) acc += g->partial[(size_t)q * g->T + t];
        g->y[(size_t)t] = acc;
    }
}

}  // namespace

extern "C" {

int sim_init(int R, int T) {
    if (R < 1 || R > 64 || T < 1) return -1;
    delete g;
    g = new Shared(R, T);
    return 0;
}

void sim_free(void) {
    delete g;
    g = nullptr;
}

// One launch over tiles 0..tiles-1 (tiles <= T: the geometry may change
// from one launch to the next): R threads, optional missing / stale
// (rank, tile).  y_out[T] receives y (NaN where no reducer wrote it).  Returns
// the status code (0 ok, 1 stale or missing flag, 2 bad ticket, 3 a rank
// gave up); *bad_tile where detected.
int sim_launch(int tiles, const double *values, unsigned seed, int skip_rank, int skip_tile, int stale_rank,
               int stale_tile, int max_sleep_us, double *y_out, int *bad_tile) {
    if (!g || tiles < 1 || tiles > g->T) return -1;
    g->status.store(0);
    g->bad_tile.store(-1);
    for (auto &v : g->y) v = std::numeric_limits<double>::quiet_NaN();
    std::vector<std::thread> th;
    for (int r = 0; r < g->R; ++r)
        th.emplace_back(rank_launch, r, tiles, values, seed * 7919u + (unsigned)r, r == skip_rank ? skip_tile : -1,
                        r == stale_rank ? stale_tile : -1, max_sleep_us);
    for (auto &t : th) t.join();
    std::memcpy(y_out, g->y.data(), sizeof(double) * (size_t)g->T);
    if (bad_tile) *bad_tile = g->bad_tile.load();
    return g->status.load();
}

// Two launches issued concurrently on the same pad, as two streams would:
// the protocol must report it, not compute garbage silently.  Returns the
// status code.
int sim_overlap(const double *values, unsigned seed) {
    if (!g) return -1;
    g->status.store(0);
    std::vector<std::thread> th;
    for (int r = 0; r < g->R; ++r) {
        th.emplace_back(rank_launch, r, g->T, values, seed + (unsigned)r, -1, -1, 50);
        th.emplace_back(rank_launch, r, g->T, values, seed + 1000u + (unsigned)r, -1, -1, 50);
    }
    for (auto &t : th) t.join();
    return g->status.load();
}

// The epoch word (the epoch of the last finished launch).
uint32_t sim_epoch(void) { return g ? g->epoch_word.load() : 0u; }

// 1 when tiles_done and every tile counter are zero (the state between
// launches), else 0.
int sim_counters_clear(void) {
    if (!g || g->tiles_done.load() != 0) return 0;
    for (auto &c : g->counters)
        if (c.load() != 0) return 0;
    return 1;
}

// The multi-GPU design's bounded wait: wait until all R flags of tile t equal
// `epoch`, giving up after timeout_us.  Returns 0, or -1 on timeout.
int sim_wait_flags(int t, uint32_t epoch, int timeout_us) {
    if (!g || t < 0 || t >= g->T) return -2;
    const auto deadline = std::chrono::steady_clock::now() + std::chrono::microseconds(timeout_us);
    while (true) {
        bool all = true;
        for (int q = 0; q < g->R; ++q)
            if (g->flags[(size_t)q * g->T + t].load(std::memory_order_acquire) != epoch) all = false;
        if (all) return 0;
        if (std::chrono::steady_clock::now() >= deadline) return -1;
        std::this_thread::yield();
    }
}

// The host's pad reset after a reported error (flags, counters and the epoch
// to zero).
void sim_reset(void) {
    if (!g) return;
    for (auto &f : g->flags) f.store(0);
    for (auto &c : g->counters) c.store(0);
    g->tiles_done.store(0);
    g->epoch_word.store(0);
}

}  // extern "C"
