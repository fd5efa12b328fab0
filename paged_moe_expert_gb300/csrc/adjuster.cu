// The adjuster: decides each scheduling round whether the expert cache in the shared page pool
// grows, shrinks or stays, which experts move, and which pages they take or give back.
//
// Rimuru, section "The adjuster: when to evict an expert, and which one?":
//   * counts: short of R_b pages -> evict ceil((R_b + 1) / 3); else fewer than 2 free pages ->
//     evict 1; else more than 9 free pages -> add min(5, floor((F_b - 9) / 3)).
//   * choice: every layer keeps the top slice of an offline ranking of its experts by routing
//     probability.  Growing, each layer nominates its next uncached expert and the most probable
//     nominees win; shrinking, each layer nominates the last expert it keeps and the least
//     probable nominees win; layers already offloading expert_offload_limit experts sit out.
//   * pages: an added expert has its pages reserved when the decision is made; an evicted
//     expert's pages are released only once the running forward pass has ended.
// Host code only: no CUDA call is made here.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>
#include <set>
#include <vector>

#include "pmoe_internal.cuh"

struct pmoe_adjuster {
    int32_t L = 0, E = 0, limit = 0;
    int64_t num_pages = 0;
    std::vector<float> prob;            // [L][E]
    std::vector<int32_t> ranking;       // [L][E]: expert at each rank, most probable first
    std::vector<int32_t> kept;          // [L]: the layer keeps ranks [0, kept)
    std::vector<int32_t> table;         // [L][E][3]: pages of W1, W3, W2, or -1
    std::set<int32_t> free_pages;       // ordered: reservations take the lowest ids
    std::vector<uint8_t> lent;          // [num_pages]: 1 while lent to the caller
    std::vector<int32_t> pending;       // (layer, expert) pairs evicted, pages not yet released
};

namespace {

// One layer's candidate for this round: its probability and the layer index.
struct Nominee {
    float p;
    int32_t layer;
};

pmoe_status bad(const char* msg) { return pmoe::record_failure(PMOE_ERR_INVALID_ARG, msg); }

}  // namespace

extern "C" pmoe_status pmoe_adjuster_create(int32_t n_layers, int32_t n_experts,
                                            const float* probs, int32_t offload_limit,
                                            const int32_t* cached, int64_t num_pages,
                                            pmoe_adjuster_t* out) {
    if (!out) return bad("pmoe_adjuster_create: out is NULL");
    *out = nullptr;
    if (n_layers < 1 || n_experts < 1 || !probs || !cached || offload_limit < 0)
        return bad("pmoe_adjuster_create: n_layers, n_experts >= 1, probs and cached non-NULL, "
                   "offload_limit >= 0");
    if (num_pages < 0 || num_pages > INT32_MAX)
        return bad("pmoe_adjuster_create: num_pages outside [0, 2^31)");
    const int64_t LE = (int64_t)n_layers * n_experts;
    int64_t need = 0;
    for (int32_t l = 0; l < n_layers; ++l) {
        if (cached[l] < 0 || cached[l] > n_experts)
            return bad("pmoe_adjuster_create: cached[l] outside [0, n_experts]");
        need += 3 * (int64_t)cached[l];
    }
    if (need > num_pages) return bad("pmoe_adjuster_create: 3 * sum(cached) > num_pages");
    for (int64_t i = 0; i < LE; ++i)
        if (!std::isfinite(probs[i])) return bad("pmoe_adjuster_create: a probability is not finite");

    pmoe_adjuster* a = new (std::nothrow) pmoe_adjuster;
    if (!a) return bad("pmoe_adjuster_create: out of host memory");
    try {
        a->L = n_layers;
        a->E = n_experts;
        a->limit = offload_limit;
        a->num_pages = num_pages;
        a->prob.assign(probs, probs + LE);
        a->ranking.resize(LE);
        a->kept.assign(cached, cached + n_layers);
        a->table.assign(LE * 3, -1);
        a->lent.assign(num_pages, 0);
        int32_t next_page = 0;
        for (int32_t l = 0; l < n_layers; ++l) {
            int32_t* r = &a->ranking[(int64_t)l * n_experts];
            const float* p = &a->prob[(int64_t)l * n_experts];
            for (int32_t e = 0; e < n_experts; ++e) r[e] = e;
            // Most probable first; equal probabilities keep the lower expert id first.
            std::stable_sort(r, r + n_experts, [p](int32_t x, int32_t y) { return p[x] > p[y]; });
            for (int32_t i = 0; i < a->kept[l]; ++i)
                for (int j = 0; j < 3; ++j)
                    a->table[((int64_t)l * n_experts + r[i]) * 3 + j] = next_page++;
        }
        for (int64_t pg = next_page; pg < num_pages; ++pg) a->free_pages.insert((int32_t)pg);
    } catch (const std::bad_alloc&) {
        delete a;
        return bad("pmoe_adjuster_create: out of host memory");
    }
    *out = a;
    return PMOE_OK;
}

extern "C" pmoe_status pmoe_adjuster_destroy(pmoe_adjuster_t adj) {
    delete adj;
    return PMOE_OK;
}

extern "C" pmoe_status pmoe_adjuster_decide(pmoe_adjuster_t a, int32_t short_pages,
                                            int32_t max_changes, int32_t* changes,
                                            int32_t* n_changes) {
    if (!a || !n_changes || short_pages < 0 || max_changes < 0 || (max_changes > 0 && !changes))
        return bad("pmoe_adjuster_decide: adjuster and n_changes non-NULL, short_pages >= 0, "
                   "max_changes >= 0, changes non-NULL when max_changes > 0");
    if (!a->pending.empty())
        return bad("pmoe_adjuster_decide: the previous round's evictions wait for "
                   "pmoe_adjuster_end_forward");
    *n_changes = 0;
    const int64_t F = (int64_t)a->free_pages.size();
    int64_t n_evict = 0, n_add = 0;
    if (short_pages > 0) n_evict = ((int64_t)short_pages + 1 + 2) / 3;  // ceil((R_b + 1) / 3)
    else if (F < 2) n_evict = 1;
    else if (F > 9) n_add = std::min<int64_t>(5, (F - 9) / 3);

    const int32_t E = a->E;
    std::vector<Nominee> nom;
    nom.reserve(a->L);
    int32_t n = 0;
    if (n_evict > 0) {
        for (int32_t l = 0; l < a->L; ++l) {
            const int32_t k = a->kept[l];
            if (k == 0 || E - k >= a->limit) continue;
            nom.push_back({a->prob[(int64_t)l * E + a->ranking[(int64_t)l * E + k - 1]], l});
        }
        // Least probable first; a tie goes to the lower layer.
        std::stable_sort(nom.begin(), nom.end(),
                         [](const Nominee& x, const Nominee& y) { return x.p < y.p; });
        const int64_t take = std::min<int64_t>({n_evict, (int64_t)nom.size(), max_changes});
        for (int64_t i = 0; i < take; ++i) {
            const int32_t l = nom[i].layer;
            const int32_t e = a->ranking[(int64_t)l * E + a->kept[l] - 1];
            const int32_t* pg = &a->table[((int64_t)l * E + e) * 3];
            int32_t* rec = changes + 6 * (int64_t)n++;
            rec[0] = -1; rec[1] = l; rec[2] = e; rec[3] = pg[0]; rec[4] = pg[1]; rec[5] = pg[2];
            a->kept[l] -= 1;
            a->pending.push_back(l);
            a->pending.push_back(e);
        }
    } else if (n_add > 0) {
        for (int32_t l = 0; l < a->L; ++l) {
            const int32_t k = a->kept[l];
            if (k == E) continue;
            nom.push_back({a->prob[(int64_t)l * E + a->ranking[(int64_t)l * E + k]], l});
        }
        // Most probable first; a tie goes to the lower layer.
        std::stable_sort(nom.begin(), nom.end(),
                         [](const Nominee& x, const Nominee& y) { return x.p > y.p; });
        const int64_t take = std::min<int64_t>({n_add, (int64_t)nom.size(), max_changes,
                                                (int64_t)a->free_pages.size() / 3});
        for (int64_t i = 0; i < take; ++i) {
            const int32_t l = nom[i].layer;
            const int32_t e = a->ranking[(int64_t)l * E + a->kept[l]];
            int32_t* pg = &a->table[((int64_t)l * E + e) * 3];
            for (int j = 0; j < 3; ++j) {
                pg[j] = *a->free_pages.begin();
                a->free_pages.erase(a->free_pages.begin());
            }
            int32_t* rec = changes + 6 * (int64_t)n++;
            rec[0] = 1; rec[1] = l; rec[2] = e; rec[3] = pg[0]; rec[4] = pg[1]; rec[5] = pg[2];
            a->kept[l] += 1;
        }
    }
    *n_changes = n;
    return PMOE_OK;
}

extern "C" pmoe_status pmoe_adjuster_end_forward(pmoe_adjuster_t a) {
    if (!a) return bad("pmoe_adjuster_end_forward: adjuster is NULL");
    for (size_t i = 0; i < a->pending.size(); i += 2) {
        int32_t* pg = &a->table[((int64_t)a->pending[i] * a->E + a->pending[i + 1]) * 3];
        for (int j = 0; j < 3; ++j) {
            a->free_pages.insert(pg[j]);
            pg[j] = -1;
        }
    }
    a->pending.clear();
    return PMOE_OK;
}

extern "C" pmoe_status pmoe_adjuster_lend(pmoe_adjuster_t a, int32_t n, int32_t* pages) {
    if (!a || n < 0 || (n > 0 && !pages))
        return bad("pmoe_adjuster_lend: adjuster non-NULL, n >= 0, pages non-NULL when n > 0");
    if ((int64_t)n > (int64_t)a->free_pages.size())
        return bad("pmoe_adjuster_lend: fewer than n pages are free");
    for (int32_t i = 0; i < n; ++i) {
        pages[i] = *a->free_pages.begin();
        a->free_pages.erase(a->free_pages.begin());
        a->lent[pages[i]] = 1;
    }
    return PMOE_OK;
}

extern "C" pmoe_status pmoe_adjuster_give_back(pmoe_adjuster_t a, int32_t n,
                                               const int32_t* pages) {
    if (!a || n < 0 || (n > 0 && !pages))
        return bad("pmoe_adjuster_give_back: adjuster non-NULL, n >= 0, pages non-NULL when n > 0");
    // Check the whole list first so that a bad entry changes nothing.
    std::vector<uint8_t> seen;
    try {
        seen.assign(a->num_pages, 0);
    } catch (const std::bad_alloc&) {
        return bad("pmoe_adjuster_give_back: out of host memory");
    }
    for (int32_t i = 0; i < n; ++i) {
        const int32_t p = pages[i];
        if (p < 0 || p >= a->num_pages || !a->lent[p] || seen[p])
            return bad("pmoe_adjuster_give_back: a page is not lent out, or listed twice");
        seen[p] = 1;
    }
    for (int32_t i = 0; i < n; ++i) {
        a->lent[pages[i]] = 0;
        a->free_pages.insert(pages[i]);
    }
    return PMOE_OK;
}

extern "C" pmoe_status pmoe_adjuster_state(pmoe_adjuster_t a, int64_t* free_pages,
                                           int32_t* cached) {
    if (!a || !free_pages) return bad("pmoe_adjuster_state: adjuster and free_pages non-NULL");
    *free_pages = (int64_t)a->free_pages.size();
    if (cached) std::memcpy(cached, a->kept.data(), sizeof(int32_t) * a->L);
    return PMOE_OK;
}

extern "C" pmoe_status pmoe_adjuster_page_table(pmoe_adjuster_t a, int32_t layer,
                                                int32_t* page_table) {
    if (!a || !page_table || layer < 0 || layer >= a->L)
        return bad("pmoe_adjuster_page_table: adjuster and page_table non-NULL, layer in range");
    std::memcpy(page_table, &a->table[(int64_t)layer * a->E * 3], sizeof(int32_t) * 3 * a->E);
    return PMOE_OK;
}
