#include "host_tables.h"

#include <algorithm>
#include <climits>
#include <cmath>
#include <numeric>
#include <queue>
#include <tuple>

namespace attn_host {

namespace {
constexpr double kTwoPi = 6.283185307179586476925286766559;
constexpr int kTile = 128;
constexpr uint32_t kNoTile = 0xFFFFu;
}  // namespace

std::vector<double> rope_thetas(int D, double base) {
    std::vector<double> th(static_cast<size_t>(D / 2));
    for (int r = 0; r < D / 2; ++r) th[r] = std::pow(base, -2.0 * static_cast<double>(r) / static_cast<double>(D));
    return th;
}

std::vector<float> rope_table(int S, int D, double base, long long pos_offset) {
    const int half = D / 2;
    const std::vector<double> th = rope_thetas(D, base);
    std::vector<float> t(static_cast<size_t>(S) * half * 2);
    for (int p = 0; p < S; ++p) {
        const double pos = static_cast<double>(p + pos_offset);
        for (int r = 0; r < half; ++r) {
            const double a = pos * th[r];
            t[(static_cast<size_t>(p) * half + r) * 2 + 0] = static_cast<float>(std::cos(a));
            t[(static_cast<size_t>(p) * half + r) * 2 + 1] = static_cast<float>(std::sin(a));
        }
    }
    return t;
}

size_t rope_factor_table_floats(int S, int D) {
    const size_t half = static_cast<size_t>(D / 2);
    const size_t rows = static_cast<size_t>(rope_rows_per_pass(D));
    const size_t ntiles = static_cast<size_t>((S + kTile - 1) / kTile);
    return (ntiles + rows + 1) * half * 2;
}

std::vector<float> rope_factor_table(int S, int D, double base) {
    const int half = D / 2;
    const int rows = rope_rows_per_pass(D);
    const int ntiles = (S + kTile - 1) / kTile;
    const std::vector<double> th = rope_thetas(D, base);
    std::vector<float> t(rope_factor_table_floats(S, D));
    size_t o = 0;
    auto put = [&](double pos) {
        for (int r = 0; r < half; ++r) {
            const double a = pos * th[r];
            t[o++] = static_cast<float>(std::cos(a));
            t[o++] = static_cast<float>(std::sin(a));
        }
    };
    for (int m = 0; m < ntiles; ++m) put(static_cast<double>(m) * kTile);
    for (int rr = 0; rr < rows; ++rr) put(static_cast<double>(rr));
    put(static_cast<double>(rows));
    return t;
}

std::vector<float> rope_split_tables(int S, int D, double base, int block) {
    const int half = D / 2;
    const int ntiles = (S + block - 1) / block;
    const std::vector<double> th = rope_thetas(D, base);
    std::vector<float> t(static_cast<size_t>(ntiles + block) * half * 2);
    size_t o = 0;
    auto put = [&](double pos) {
        for (int r = 0; r < half; ++r) {
            t[o++] = static_cast<float>(std::cos(pos * th[r]));
            t[o++] = static_cast<float>(std::sin(pos * th[r]));
        }
    };
    for (int m = 0; m < ntiles; ++m) put(static_cast<double>(m) * block);
    for (int rr = 0; rr < block; ++rr) put(static_cast<double>(rr));
    return t;
}

std::vector<int32_t> window_widths(int D, double base, double k) {
    std::vector<int32_t> w(static_cast<size_t>(D / 2), INT32_MAX);
    if (!(k > 0.0) || std::isinf(k)) return w;
    const std::vector<double> th = rope_thetas(D, base);
    for (int r = 0; r < D / 2; ++r) {
        const double x = std::floor(k * kTwoPi / th[r]);
        w[r] = x >= static_cast<double>(INT32_MAX) ? INT32_MAX : static_cast<int32_t>(std::max(0.0, x));
    }
    return w;
}

std::vector<int16_t> window_tile_table(int S, int D, double base, double k) {
    const std::vector<int32_t> w = window_widths(D, base, k);
    const int ntiles = (S + kTile - 1) / kTile;
    auto first = [&](long long d) {
        int r = 0;
        while (r < D / 2 && static_cast<long long>(w[r]) < d) ++r;
        return static_cast<int16_t>(r);
    };
    std::vector<int16_t> t(static_cast<size_t>(ntiles) * 2);
    for (int i = 0; i < ntiles; ++i) {
        t[2 * i] = first(std::max<long long>(0, static_cast<long long>(kTile) * i - (kTile - 1)));
        t[2 * i + 1] = first(static_cast<long long>(kTile) * i + (kTile - 1));
    }
    return t;
}

long long schedule_units(int B, int Hq, int Hkv, int S) {
    const long long nqt = (S + kTile - 1) / kTile;
    const long long G = Hq / Hkv;
    if (G >= 2) return static_cast<long long>(B) * Hkv * nqt * ((G + 1) / 2);
    return static_cast<long long>(B) * Hq * ((nqt + 1) / 2);
}

Schedule build_schedule(int B, int Hq, int Hkv, int S, int D, bool causal, int num_ctas, double kv_window_bytes) {
    struct U {
        uint32_t x, y;
        double cost;
        int kv;  // b * Hkv + KV head: the window key
    };
    const int nqt = (S + kTile - 1) / kTile;
    const int G = Hq / Hkv;
    auto tile_cost = [&](int qt) { return 2.0 * ((causal ? qt : nqt - 1) + 1); };
    std::vector<U> units;
    if (G >= 2) {
        // two query heads of one KV group at the same query tile
        for (int b = 0; b < B; ++b)
            for (int g = 0; g < Hkv; ++g)
                for (int qt = 0; qt < nqt; ++qt)
                    for (int h = g * G; h < (g + 1) * G; h += 2) {
                        const bool pair = h + 1 < (g + 1) * G;
                        U u;
                        u.x = static_cast<uint32_t>(qt) | ((pair ? static_cast<uint32_t>(qt) : kNoTile) << 16);
                        u.y = static_cast<uint32_t>(h) | (static_cast<uint32_t>(pair ? h + 1 : h) << 8) |
                              (static_cast<uint32_t>(b) << 16);
                        u.cost = tile_cost(qt) * (pair ? 2 : 1) + 4.0;
                        u.kv = b * Hkv + g;
                        units.push_back(u);
                    }
    } else {
        // two consecutive query tiles of one head
        for (int b = 0; b < B; ++b)
            for (int h = 0; h < Hq; ++h)
                for (int t = 0; 2 * t < nqt; ++t) {
                    const int q0 = 2 * t, q1 = 2 * t + 1;
                    const bool pair = q1 < nqt;
                    U u;
                    u.x = static_cast<uint32_t>(q0) | ((pair ? static_cast<uint32_t>(q1) : kNoTile) << 16);
                    u.y = static_cast<uint32_t>(h) | (static_cast<uint32_t>(h) << 8) | (static_cast<uint32_t>(b) << 16);
                    u.cost = tile_cost(q0) + (pair ? tile_cost(q1) : 0.0) + 4.0;
                    u.kv = b * Hkv + h;
                    units.push_back(u);
                }
    }
    Schedule sc;
    const int n = static_cast<int>(units.size());
    sc.ctas = std::max(1, std::min(num_ctas, n));
    // KV heads per window: K and V of one KV head take 2 * 2 * S * D bytes (bf16)
    const double kv_head_bytes = 4.0 * static_cast<double>(S) * static_cast<double>(D);
    const long long kv_heads = static_cast<long long>(B) * Hkv;
    // KV heads per window (all of them without a window size).  The last window evens out the loads
    // that the earlier ones leave, so it takes at least three units per CTA; the heads before it are
    // split into windows whose sizes differ by at most one head.
    long long cap = kv_heads;
    if (kv_window_bytes > 0.0)
        cap = std::max<long long>(1, std::min<long long>(kv_heads, static_cast<long long>(kv_window_bytes / kv_head_bytes)));
    const long long units_per_kv = (n + kv_heads - 1) / kv_heads;
    const long long tail_heads =
        std::min<long long>(kv_heads, std::max<long long>(cap, (3LL * sc.ctas + units_per_kv - 1) / units_per_kv));
    const long long front_heads = kv_heads - tail_heads;
    const long long front_windows = (front_heads + cap - 1) / cap;
    auto window_of = [&](int kv) -> long long {
        if (kv >= front_heads) return front_windows;
        return static_cast<long long>(kv) * front_windows / front_heads;
    };
    // window by window; inside a window, heaviest first (stable: ties keep the (batch, head, tile) order)
    std::vector<int> order(n);
    std::iota(order.begin(), order.end(), 0);
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
        const long long wa = window_of(units[a].kv), wb = window_of(units[b].kv);
        if (wa != wb) return wa < wb;
        return units[a].cost > units[b].cost;
    });
    using Load = std::pair<double, int>;
    std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
    for (int c = 0; c < sc.ctas; ++c) heap.push({0.0, c});
    std::vector<std::vector<int>> bins(sc.ctas);
    std::vector<double> load(sc.ctas, 0.0);
    for (int i : order) {
        Load top = heap.top();
        heap.pop();
        bins[top.second].push_back(i);
        top.first += units[i].cost;
        load[top.second] = top.first;
        heap.push(top);
    }
    sc.offsets.push_back(0);
    for (int c = 0; c < sc.ctas; ++c) {
        for (int i : bins[c]) {
            sc.words.push_back(units[i].x);
            sc.words.push_back(units[i].y);
        }
        sc.offsets.push_back(static_cast<int32_t>(sc.words.size() / 2));
    }
    sc.max_cost = *std::max_element(load.begin(), load.end());
    sc.mean_cost = std::accumulate(load.begin(), load.end(), 0.0) / sc.ctas;
    return sc;
}

MaskSchedule build_mask_schedule(const int* row_ptr, int nrows, long long bh, int num_ctas) {
    MaskSchedule sc;
    const long long n = static_cast<long long>(nrows) * bh;
    sc.ctas = static_cast<int>(std::max<long long>(1, std::min<long long>(num_ctas, (n + 1) / 2)));
    const int nbins = 2 * sc.ctas;  // two task streams per CTA
    // rows of tiles by cost, heaviest first; every batch-head of a row costs the same
    std::vector<int> rows(nrows);
    std::iota(rows.begin(), rows.end(), 0);
    auto cost = [&](int i) { return static_cast<double>(row_ptr[i + 1] - row_ptr[i]) + kMaskTileFixedCost; };
    std::stable_sort(rows.begin(), rows.end(), [&](int a, int b) { return cost(a) > cost(b); });
    using Load = std::pair<double, int>;
    std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
    for (int c = 0; c < nbins; ++c) heap.push({0.0, c});
    std::vector<std::vector<int32_t>> bins(nbins);
    for (int i : rows)
        for (long long x = 0; x < bh; ++x) {
            Load top = heap.top();
            heap.pop();
            bins[top.second].push_back(static_cast<int32_t>(i * bh + x));
            top.first += cost(i);
            heap.push(top);
        }
    // each stream runs its tasks by (batch-head, descending query tile): all streams sweep the
    // batch-heads in the same order, so the streams running at one time share K/V tiles in L2
    for (auto& bin : bins)
        std::stable_sort(bin.begin(), bin.end(), [&](int32_t a, int32_t b) {
            return std::make_pair(a % bh, -(a / bh)) < std::make_pair(b % bh, -(b / bh));
        });
    sc.offsets.push_back(0);
    for (auto& bin : bins) {
        sc.tasks.insert(sc.tasks.end(), bin.begin(), bin.end());
        sc.offsets.push_back(static_cast<int32_t>(sc.tasks.size()));
    }
    return sc;
}

}  // namespace attn_host
