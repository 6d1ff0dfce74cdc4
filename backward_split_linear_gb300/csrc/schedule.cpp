// F/B/W order of one pipeline stage (CPU only) and the unit-time pipeline model.
//
// "Zero-Bubble Pipeline Parallelism Guide for LLMs":
//  - section "2. The 1F1B (One-Forward-One-Backward) Schedule" and the first
//    diagram of "The Mechanics of Pipeline Bubbles": stage s runs p - s
//    forwards before its first backward, then alternates B and F;
//  - section "Core Innovation 2" (ZB-1F1B, here ZB-H1): same activation memory
//    as 1F1B, F and B keep priority, a W fills each slot that would idle, the
//    steady state runs F -> B -> W, leftover W drain at the end;
//  - section "Memory Management & Activation Rollback": at the in-flight
//    ceiling a W must run before the next F;
//  - section "Mathematical Modeling": unit op times, bubble formulas.
//
// ZB-2p (section "Core Innovation 2", item 2): the same policy with a ceiling
// of 2p held microbatches and 2(p-s)-1 forwards before the first B of stage
// s; every stage then works without idle from its first op to its last when
// m >= 2p - 1.  Emitted by a step-by-step run of the policy.
//
// Memory-limited orders ("Zero Bubble Pipeline Parallelism", abstract: a
// search for the best schedule under a memory limit; the guide: ZB-H1 holds
// p microbatches, ZB-2p 2p): the same policy with a ceiling L in [p, 2p] and
// min(L - s, 2(p - s) - 1) forwards before the first B of stage s, run with
// measured op durations; zb_schedule_search takes the L within the memory
// limit whose run ends first.
//
// ZB-H1, m >= p, in closed form for stage s:
//   F_0 .. F_{p-s-1}
//   B_j, F_{p-s+j}            for j = 0 .. s-1
//   B_{s+k}, W_k, F_{p+k}     for k = 0 .. m-p-1     (steady F -> B -> W)
//   B_{s+k}, W_k              for k = m-p .. m-s-1
//   W_k                       for k = m-s .. m-1     (drain)
// It keeps the 1F1B F/B order, never holds more than p microbatches and ends
// every stage at 3m + p - 1 units.  For m < p the same policy is run step by
// step over all stages instead.
#include <algorithm>
#include <vector>

#include "../../include/zb.h"

namespace {

struct Op {
    char kind;
    int mb;
};

void order_gpipe(int, int, int m, std::vector<Op>& o) {
    for (int i = 0; i < m; ++i) o.push_back({'F', i});
    for (int i = 0; i < m; ++i) {
        o.push_back({'B', i});
        o.push_back({'W', i});
    }
}

void order_1f1b(int s, int p, int m, std::vector<Op>& o) {
    const int warm = std::min(p - s - 1, m);
    for (int i = 0; i < warm; ++i) o.push_back({'F', i});
    for (int j = 0; j < m - warm; ++j) {
        o.push_back({'F', warm + j});
        o.push_back({'B', j});
        o.push_back({'W', j});
    }
    for (int i = m - warm; i < m; ++i) {
        o.push_back({'B', i});
        o.push_back({'W', i});
    }
}

void order_zbh1_closed(int s, int p, int m, std::vector<Op>& o) {
    for (int i = 0; i < p - s; ++i) o.push_back({'F', i});
    for (int j = 0; j < s; ++j) {
        o.push_back({'B', j});
        o.push_back({'F', p - s + j});
    }
    for (int k = 0; k < m - p; ++k) {
        o.push_back({'B', s + k});
        o.push_back({'W', k});
        o.push_back({'F', p + k});
    }
    for (int k = m - p; k < m - s; ++k) {
        o.push_back({'B', s + k});
        o.push_back({'W', k});
    }
    for (int k = m - s; k < m; ++k) o.push_back({'W', k});
}

// F/B order of stage s: `warm` forwards, then B and F alternate, then the last B.
void fb_order(int warm, int m, std::vector<Op>& o) {
    warm = std::min(warm, m);
    for (int i = 0; i < warm; ++i) o.push_back({'F', i});
    for (int j = 0; j < m - warm; ++j) {
        o.push_back({'B', j});
        o.push_back({'F', warm + j});
    }
    for (int i = m - warm; i < m; ++i) o.push_back({'B', i});
}

// Step-by-step run of the ZB-H1 policy on all p stages.  At every unit of
// time each free stage, looking at the state at that time: runs its next F/B
// if that op's inputs exist, unless it is an F that would pass the ceiling of
// `limit` held microbatches, in which case it runs its oldest pending W; if
// the next F/B is not ready it runs the oldest pending W; else it idles.
// Stage s runs warm(s) forwards before its first B: p - s for ZB-H1 (the 1F1B
// order), 2(p - s) - 1 for ZB-2p.
std::vector<std::vector<Op>> zb_policy_all(int p, int m, int limit, bool two_p) {
    std::vector<std::vector<Op>> fb(p), out(p);
    for (int s = 0; s < p; ++s) fb_order(two_p ? 2 * (p - s) - 1 : p - s, m, fb[s]);
    // finish time of F/B per (stage, mb); -1 = not run
    std::vector<int> fin_f(p * m, -1), fin_b(p * m, -1);
    std::vector<size_t> ptr(p, 0);
    std::vector<int> held(p, 0), busy(p, 0);
    std::vector<std::vector<int>> pending(p);
    int done = 0;
    const int total = 3 * m * p;
    for (int t = 0; done < total && t < 64 * (m + p) + 64; ++t) {
        std::vector<Op> choice(p, Op{0, -1});
        for (int s = 0; s < p; ++s) {
            if (busy[s] > t) continue;
            if (ptr[s] < fb[s].size()) {
                const Op nx = fb[s][ptr[s]];
                bool ready;
                if (nx.kind == 'F')
                    ready = s == 0 || (fin_f[(s - 1) * m + nx.mb] >= 0 && fin_f[(s - 1) * m + nx.mb] <= t);
                else
                    ready = fin_f[s * m + nx.mb] >= 0 && fin_f[s * m + nx.mb] <= t &&
                            (s == p - 1 || (fin_b[(s + 1) * m + nx.mb] >= 0 && fin_b[(s + 1) * m + nx.mb] <= t));
                if (ready) {
                    if (nx.kind == 'F' && held[s] >= limit) {
                        if (!pending[s].empty()) choice[s] = {'W', pending[s].front()};
                    } else {
                        choice[s] = nx;
                    }
                } else if (!pending[s].empty()) {
                    choice[s] = {'W', pending[s].front()};
                }
            } else if (!pending[s].empty()) {
                choice[s] = {'W', pending[s].front()};
            }
        }
        for (int s = 0; s < p; ++s) {
            const Op op = choice[s];
            if (op.mb < 0) continue;
            busy[s] = t + 1;
            out[s].push_back(op);
            ++done;
            if (op.kind == 'W') {
                pending[s].erase(pending[s].begin());
                --held[s];
            } else {
                ++ptr[s];
                if (op.kind == 'F') {
                    fin_f[s * m + op.mb] = t + 1;
                    ++held[s];
                } else {
                    fin_b[s * m + op.mb] = t + 1;
                    pending[s].push_back(op.mb);
                }
            }
        }
    }
    return out;
}

// The same policy with op durations t_f, t_b, t_w: stages decide whenever
// they are free, all on the state at that moment; time then jumps to the next
// end of an op.  warm[s] forwards precede stage s's first B.  Returns false
// (and leaves `out` incomplete) if the run cannot go on.
bool zb_policy_timed(int p, int m, int limit, const std::vector<int>& warm, long long t_f, long long t_b,
                     long long t_w, std::vector<std::vector<Op>>& out, long long* span) {
    std::vector<std::vector<Op>> fb(p);
    out.assign(p, {});
    for (int s = 0; s < p; ++s) fb_order(warm[s], m, fb[s]);
    std::vector<long long> fin_f(static_cast<size_t>(p) * m, -1), fin_b(static_cast<size_t>(p) * m, -1);
    std::vector<size_t> ptr(p, 0);
    std::vector<int> held(p, 0);
    std::vector<long long> busy(p, 0);
    std::vector<std::vector<int>> pending(p);
    long long done = 0, t = 0, end = 0;
    const long long total = 3LL * m * p;
    std::vector<Op> choice(p);
    while (done < total) {
        for (int s = 0; s < p; ++s) {
            choice[s] = Op{0, -1};
            if (busy[s] > t) continue;
            if (ptr[s] < fb[s].size()) {
                const Op nx = fb[s][ptr[s]];
                bool ready;
                if (nx.kind == 'F') {
                    const long long d = s == 0 ? 0 : fin_f[static_cast<size_t>(s - 1) * m + nx.mb];
                    ready = d >= 0 && d <= t;
                } else {
                    const long long f = fin_f[static_cast<size_t>(s) * m + nx.mb];
                    const long long b = s == p - 1 ? 0 : fin_b[static_cast<size_t>(s + 1) * m + nx.mb];
                    ready = f >= 0 && f <= t && b >= 0 && b <= t;
                }
                if (ready) {
                    if (nx.kind == 'F' && held[s] >= limit) {
                        if (!pending[s].empty()) choice[s] = {'W', pending[s].front()};
                    } else {
                        choice[s] = nx;
                    }
                } else if (!pending[s].empty()) {
                    choice[s] = {'W', pending[s].front()};
                }
            } else if (!pending[s].empty()) {
                choice[s] = {'W', pending[s].front()};
            }
        }
        for (int s = 0; s < p; ++s) {
            const Op op = choice[s];
            if (op.mb < 0) continue;
            const long long d = op.kind == 'F' ? t_f : (op.kind == 'B' ? t_b : t_w);
            busy[s] = t + d;
            end = std::max(end, t + d);
            out[s].push_back(op);
            ++done;
            if (op.kind == 'W') {
                pending[s].erase(pending[s].begin());
                --held[s];
            } else {
                ++ptr[s];
                if (op.kind == 'F') {
                    fin_f[static_cast<size_t>(s) * m + op.mb] = t + d;
                    ++held[s];
                } else {
                    fin_b[static_cast<size_t>(s) * m + op.mb] = t + d;
                    pending[s].push_back(op.mb);
                }
            }
        }
        if (done == total) break;
        long long next = -1;
        for (int s = 0; s < p; ++s)
            if (busy[s] > t && (next < 0 || busy[s] < next)) next = busy[s];
        if (next < 0) return false;
        t = next;
    }
    *span = end;
    return true;
}

void stage_order(zb_sched_kind kind, int s, int p, int m, std::vector<Op>& o) {
    if (kind == ZB_SCHED_GPIPE) {
        order_gpipe(s, p, m, o);
    } else if (kind == ZB_SCHED_1F1B) {
        order_1f1b(s, p, m, o);
    } else if (kind == ZB_SCHED_ZB2P) {
        o = zb_policy_all(p, m, 2 * p, true)[s];
    } else if (m >= p) {
        order_zbh1_closed(s, p, m, o);
    } else {
        o = zb_policy_all(p, m, p, false)[s];
    }
}

bool valid_kind(int k) {
    return k == ZB_SCHED_1F1B || k == ZB_SCHED_ZBH1 || k == ZB_SCHED_GPIPE || k == ZB_SCHED_ZB2P;
}

}  // namespace

extern "C" zb_status zb_schedule(zb_sched_kind kind, int32_t stage, int32_t p, int32_t m, zb_op* out,
                                 int32_t cap, int32_t* n_out) {
    if (!valid_kind(kind) || p < 1 || m < 1 || stage < 0 || stage >= p || !n_out ||
        (cap > 0 && !out) || cap < 0 || m > (1 << 24))
        return ZB_ERR_ARG;
    *n_out = 3 * m;
    if (cap < 3 * m) return ZB_ERR_CAPACITY;
    std::vector<Op> o;
    o.reserve(3 * m);
    stage_order(kind, stage, p, m, o);
    if (o.size() != static_cast<size_t>(3 * m)) return ZB_ERR_ORDER;  // policy run did not finish
    for (int i = 0; i < 3 * m; ++i) {
        out[i].kind = static_cast<uint8_t>(o[i].kind);
        out[i].pad[0] = out[i].pad[1] = out[i].pad[2] = 0;
        out[i].mb = o[i].mb;
    }
    return ZB_OK;
}

// Unit-time run of the p stages' orders: finish time of every op's stage
// window, and the makespan.  Returns false if the orders deadlock.
namespace {
bool run_unit_model(zb_sched_kind kind, int p, int m, int* span_out, long long* window_idle_out) {
    const bool split = kind == ZB_SCHED_ZBH1 || kind == ZB_SCHED_ZB2P;
    std::vector<std::vector<Op>> orders(p);
    for (int s = 0; s < p; ++s) {
        stage_order(kind, s, p, m, orders[s]);
        if (orders[s].size() != static_cast<size_t>(3 * m)) return false;
    }
    auto idx = [m](int s, int i) { return s * m + i; };
    std::vector<int> ff(p * m, -1), fb(p * m, -1), fw(p * m, -1);
    std::vector<size_t> ptr(p, 0);
    std::vector<int> free_at(p, 0), first(p, -1), last(p, 0);
    size_t placed = 0, total = static_cast<size_t>(3) * m * p;
    int span = 0;
    while (placed < total) {
        bool progressed = false;
        for (int s = 0; s < p; ++s) {
            while (ptr[s] < orders[s].size()) {
                const Op op = orders[s][ptr[s]];
                int ready = free_at[s];
                bool ok = true;
                if (op.kind == 'F') {
                    if (s > 0) {
                        const int d = ff[idx(s - 1, op.mb)];
                        ok = d >= 0;
                        ready = std::max(ready, d);
                    }
                } else if (op.kind == 'B') {
                    const int d0 = ff[idx(s, op.mb)];
                    ok = d0 >= 0;
                    ready = std::max(ready, d0);
                    if (s < p - 1) {
                        const int d1 = split ? fb[idx(s + 1, op.mb)] : fw[idx(s + 1, op.mb)];
                        ok = ok && d1 >= 0;
                        ready = std::max(ready, d1);
                    }
                } else {
                    const int d = fb[idx(s, op.mb)];
                    ok = d >= 0;
                    ready = std::max(ready, d);
                }
                if (!ok) break;
                const int fin = ready + 1;
                (op.kind == 'F' ? ff : op.kind == 'B' ? fb : fw)[idx(s, op.mb)] = fin;
                if (first[s] < 0) first[s] = ready;
                last[s] = fin;
                free_at[s] = fin;
                span = std::max(span, fin);
                ++ptr[s];
                ++placed;
                progressed = true;
            }
        }
        if (!progressed) return false;
    }
    long long window_idle = 0;
    for (int s = 0; s < p; ++s) window_idle += (last[s] - first[s]) - 3LL * m;
    *span_out = span;
    *window_idle_out = window_idle;
    return true;
}
}  // namespace

extern "C" zb_status zb_schedule_window_idle(zb_sched_kind kind, int32_t p, int32_t m, int64_t* idle_units,
                                             double* idle_over_compute) {
    if (!valid_kind(kind) || p < 1 || m < 1 || p > 4096 || m > (1 << 20)) return ZB_ERR_ARG;
    int span = 0;
    long long idle = 0;
    if (!run_unit_model(kind, p, m, &span, &idle)) return ZB_ERR_ORDER;
    if (idle_units) *idle_units = idle;
    if (idle_over_compute) *idle_over_compute = static_cast<double>(idle) / (3.0 * m * p);
    return ZB_OK;
}

extern "C" zb_status zb_schedule_bubble(zb_sched_kind kind, int32_t p, int32_t m, int32_t* makespan,
                                        double* idle_over_compute, double* idle_over_wall) {
    if (!valid_kind(kind) || p < 1 || m < 1 || p > 4096 || m > (1 << 20)) return ZB_ERR_ARG;
    int span = 0;
    long long window_idle = 0;
    if (!run_unit_model(kind, p, m, &span, &window_idle)) return ZB_ERR_ORDER;
    const double compute = 3.0 * m * p;
    const double idle = static_cast<double>(p) * span - compute;
    if (makespan) *makespan = span;
    if (idle_over_compute) *idle_over_compute = idle / compute;
    if (idle_over_wall) *idle_over_wall = idle / (static_cast<double>(p) * span);
    return ZB_OK;
}

extern "C" zb_status zb_schedule_search(int32_t stage, int32_t p, int32_t m, int32_t mem_limit, int32_t t_f,
                                        int32_t t_b, int32_t t_w, zb_op* out, int32_t cap, int32_t* n_out,
                                        int32_t* chosen_limit, int64_t* makespan) {
    if (p < 1 || m < 1 || stage < 0 || stage >= p || !n_out || (cap > 0 && !out) || cap < 0 || mem_limit < p ||
        t_f < 1 || t_b < 1 || t_w < 1 || static_cast<long long>(p) * m > (1LL << 20))
        return ZB_ERR_ARG;
    *n_out = 3 * m;
    if (cap < 3 * m) return ZB_ERR_CAPACITY;
    int best_limit = -1;
    long long best_span = -1;
    std::vector<std::vector<Op>> best, cur;
    const int top = std::min(2 * p, mem_limit);
    for (int limit = p; limit <= top; ++limit) {
        std::vector<int> warm(p);
        for (int s = 0; s < p; ++s) warm[s] = std::min(limit - s, 2 * (p - s) - 1);
        long long span = 0;
        if (!zb_policy_timed(p, m, limit, warm, t_f, t_b, t_w, cur, &span)) return ZB_ERR_ORDER;
        if (best_limit < 0 || span < best_span) {
            best_limit = limit;
            best_span = span;
            best.swap(cur);
        }
    }
    const std::vector<Op>& o = best[stage];
    if (o.size() != static_cast<size_t>(3 * m)) return ZB_ERR_ORDER;
    for (int i = 0; i < 3 * m; ++i) {
        out[i].kind = static_cast<uint8_t>(o[i].kind);
        out[i].pad[0] = out[i].pad[1] = out[i].pad[2] = 0;
        out[i].mb = o[i].mb;
    }
    if (chosen_limit) *chosen_limit = best_limit;
    if (makespan) *makespan = best_span;
    return ZB_OK;
}
