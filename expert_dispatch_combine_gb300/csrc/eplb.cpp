// eplb.cpp -- EPLB replica planner (host).
//
// "xDeepServe on CloudMatrix384", section "专家负载均衡":
//   P069-P075  greedy selection: per time slice the hot expert is the arg-max
//              of token_count; the tail load is the sum over slices of the hot
//              load; each round every candidate (hot in some slice) is tried
//              with its tokens split evenly over one more copy, and the one
//              giving the smallest tail load is taken and applied;
//   P076       placement, heaviest replica first, on the least-loaded rank
//              that still has a free redundant slot.
// Readings where the page is silent: ties go to the lower expert id / rank;
// a replica's share is total/instances; a rank's starting load is the sum of
// its primary experts' shares; a rank already hosting the expert is skipped
// while another rank has a free slot; replica lists are in ascending
// physical id.
#include <algorithm>
#include <limits>
#include <vector>

#include "moe.h"

extern "C" moe_status moe_eplb_plan(int32_t n_slices, int32_t E_log, int32_t E_phys,
                                    int32_t n_ranks, const double* token_count,
                                    int32_t max_copies, int32_t* rep_table, int32_t* n_copies,
                                    int32_t* phys_to_logical) {
    if (n_slices < 1 || E_log < 1 || n_ranks < 1 || E_phys < E_log || E_log % n_ranks ||
        E_phys % n_ranks || !token_count || !rep_table || !n_copies || !phys_to_logical ||
        max_copies < 1)
        return MOE_ERR_INVALID_ARG;
    const int E = E_log, NS = n_slices;
    const int budget = E_phys - E_log;
    auto tc = [&](int t, int e) { return token_count[(size_t)t * E + e]; };

    // ---- selection
    std::vector<int> copies(E, 1);
    std::vector<double> sim((size_t)NS * E);
    for (int t = 0; t < NS; ++t)
        for (int e = 0; e < E; ++e) sim[(size_t)t * E + e] = tc(t, e);
    std::vector<int> replicas;
    std::vector<char> is_cand(E);
    for (int round = 0; round < budget; ++round) {
        std::fill(is_cand.begin(), is_cand.end(), 0);
        for (int t = 0; t < NS; ++t) {
            int h = 0;
            for (int e = 1; e < E; ++e)
                if (sim[(size_t)t * E + e] > sim[(size_t)t * E + h]) h = e;
            is_cand[h] = 1;
        }
        int best = -1;
        double best_tail = std::numeric_limits<double>::infinity();
        for (int c = 0; c < E; ++c) {
            if (!is_cand[c]) continue;
            double tail = 0.0;
            for (int t = 0; t < NS; ++t) {
                double m = -std::numeric_limits<double>::infinity();
                for (int e = 0; e < E; ++e) {
                    double v = (e == c) ? tc(t, c) / (double)(copies[c] + 1) : sim[(size_t)t * E + e];
                    if (v > m) m = v;
                }
                tail += m;
            }
            if (tail < best_tail) { best = c; best_tail = tail; }
        }
        if (best < 0) break;
        replicas.push_back(best);
        copies[best] += 1;
        for (int t = 0; t < NS; ++t) sim[(size_t)t * E + best] = tc(t, best) / (double)copies[best];
    }

    // ---- placement
    const int R = n_ranks, ppr = E / R, epr = E_phys / R, rpr = epr - ppr;
    std::vector<double> total(E, 0.0);
    for (int e = 0; e < E; ++e) {
        double s = 0.0;
        for (int t = 0; t < NS; ++t) s += tc(t, e);
        total[e] = s;
    }
    std::vector<double> load(R, 0.0);
    std::vector<int> freeslots(R, rpr);
    std::vector<std::vector<char>> hosts(R, std::vector<char>(E, 0));
    for (int p = 0; p < E_phys; ++p) phys_to_logical[p] = -1;
    for (int r = 0; r < R; ++r)
        for (int m = 0; m < ppr; ++m) {
            int e = r * ppr + m;
            phys_to_logical[r * epr + m] = e;
            hosts[r][e] = 1;
            load[r] += total[e] / (double)copies[e];
        }
    std::vector<int> ordered = replicas;
    std::stable_sort(ordered.begin(), ordered.end(), [&](int a, int b) {
        if (total[a] != total[b]) return total[a] > total[b];
        return a < b;
    });
    for (int e : ordered) {
        int tgt = -1;
        for (int pass = 0; pass < 2 && tgt < 0; ++pass) {
            for (int r = 0; r < R; ++r) {
                if (freeslots[r] <= 0) continue;
                if (pass == 0 && hosts[r][e]) continue;
                if (tgt < 0 || load[r] < load[tgt]) tgt = r;
            }
        }
        if (tgt < 0) return MOE_ERR_INVALID_ARG;  // unreachable: budget == free slots
        int slot = tgt * epr + ppr + (rpr - freeslots[tgt]);
        freeslots[tgt] -= 1;
        phys_to_logical[slot] = e;
        hosts[tgt][e] = 1;
        load[tgt] += total[e] / (double)copies[e];
    }

    // ---- replica lists, ascending physical id
    std::vector<std::vector<int>> lists(E);
    for (int p = 0; p < E_phys; ++p)
        if (phys_to_logical[p] >= 0) lists[phys_to_logical[p]].push_back(p);
    for (int e = 0; e < E; ++e)
        if ((int)lists[e].size() > max_copies) return MOE_ERR_INVALID_ARG;
    for (int e = 0; e < E; ++e) {
        n_copies[e] = (int32_t)lists[e].size();
        for (int c = 0; c < max_copies; ++c)
            rep_table[(size_t)e * max_copies + c] = c < (int)lists[e].size() ? lists[e][c] : -1;
    }
    return MOE_OK;
}
