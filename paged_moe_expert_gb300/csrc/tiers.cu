// Three tiers of pages over one pool: huge pages split into expert / SSM pages, expert pages split
// into KV cache / convolution-state pages, and both merge back when their parts are all free.
// Rimuru, section "One pool for data whose sizes differ by orders of magnitude".  Host code only.
#include <map>
#include <numeric>
#include <set>
#include <vector>

#include "pmoe_internal.cuh"

namespace {

constexpr int kNoKind = -1;

// A huge page: whole, or split into middle pages of one kind.
struct Huge {
    int kind = kNoKind;     // PMOE_PAGE_EXPERT / PMOE_PAGE_SSM once split
    int live = 0;           // middle pages in use (live or split into small pages)
};

// An expert page split into small pages of one kind.
struct Split {
    int kind = kNoKind;               // PMOE_PAGE_KV / PMOE_PAGE_CONV
    std::vector<int64_t> owner;       // per slot: owner of the live small page, or -1
    int live = 0;
};

}  // namespace

struct pmoe_tiers {
    int64_t huge_bytes = 0, size[4] = {0, 0, 0, 0};
    int64_t n_huge = 0;
    std::vector<Huge> huge;
    std::set<int64_t> free_huge;                  // huge page indices
    std::set<int64_t> free_mid[2];                // byte offsets of free expert / SSM pages
    std::set<int64_t> live_mid[2];                // byte offsets of middle pages handed out
    std::map<int64_t, Split> split;               // expert page offset -> its small pages
    std::set<int64_t> has_free[2];                // split pages (offsets) of kind KV / CONV with a free slot
    std::map<int64_t, std::map<int64_t, int>> by_owner[2];   // owner -> split page -> its live slots
};

namespace {

pmoe_status bad(const char* msg) { return pmoe::record_failure(PMOE_ERR_INVALID_ARG, msg); }

int64_t gcd64(int64_t a, int64_t b) { return b == 0 ? a : gcd64(b, a % b); }

// A middle page of `kind` (0 expert, 1 SSM): a free one, else the lowest free huge page split.
int64_t take_mid(pmoe_tiers* t, int kind) {
    std::set<int64_t>& fr = t->free_mid[kind];
    if (fr.empty()) {
        if (t->free_huge.empty()) return -1;
        const int64_t h = *t->free_huge.begin();
        t->free_huge.erase(t->free_huge.begin());
        t->huge[h].kind = kind;
        t->huge[h].live = 0;
        const int64_t per = t->huge_bytes / t->size[kind];
        for (int64_t i = 0; i < per; ++i) fr.insert(h * t->huge_bytes + i * t->size[kind]);
    }
    const int64_t off = *fr.begin();
    fr.erase(fr.begin());
    t->huge[off / t->huge_bytes].live += 1;
    return off;
}

// A middle page back: free, and the huge page whole again once all its middle pages are free.
void give_mid(pmoe_tiers* t, int kind, int64_t off) {
    const int64_t h = off / t->huge_bytes;
    t->free_mid[kind].insert(off);
    if (--t->huge[h].live == 0) {
        const int64_t per = t->huge_bytes / t->size[kind];
        for (int64_t i = 0; i < per; ++i) t->free_mid[kind].erase(h * t->huge_bytes + i * t->size[kind]);
        t->huge[h].kind = kNoKind;
        t->free_huge.insert(h);
    }
}

int64_t take_small(pmoe_tiers* t, int kind, int64_t owner) {
    const int s = kind - PMOE_PAGE_KV;
    std::set<int64_t>& cand = t->has_free[s];
    int64_t page = -1;
    auto mine = t->by_owner[s].find(owner);
    if (mine != t->by_owner[s].end())   // a split page that already holds this owner's pages
        for (const auto& pc : mine->second)
            if (cand.count(pc.first)) { page = pc.first; break; }
    if (page < 0 && !cand.empty()) page = *cand.begin();
    if (page < 0) {                    // split an expert page for it
        const int64_t e = take_mid(t, PMOE_PAGE_EXPERT);
        if (e < 0) return -1;
        Split sp;
        sp.kind = kind;
        sp.owner.assign(t->size[PMOE_PAGE_EXPERT] / t->size[kind], -1);
        t->split[e] = sp;
        cand.insert(e);
        page = e;
    }
    Split& sp = t->split[page];
    int64_t slot = 0;
    while (sp.owner[slot] >= 0) ++slot;
    sp.owner[slot] = owner;
    sp.live += 1;
    t->by_owner[s][owner][page] += 1;
    if (sp.live == (int)sp.owner.size()) cand.erase(page);
    return page + slot * t->size[kind];
}

}  // namespace

extern "C" pmoe_status pmoe_tiers_create(int64_t pool_bytes, int64_t expert_page, int64_t ssm_page,
                                         int64_t kv_page, int64_t conv_page, pmoe_tiers_t* out) {
    if (!out) return bad("pmoe_tiers_create: out is NULL");
    *out = nullptr;
    if (pool_bytes < 0 || expert_page <= 0 || ssm_page < 0 || kv_page < 0 || conv_page < 0)
        return bad("pmoe_tiers_create: sizes must be >= 0 and expert_page > 0");
    if ((kv_page && expert_page % kv_page) || (conv_page && expert_page % conv_page))
        return bad("pmoe_tiers_create: small page sizes must divide the expert page");
    int64_t huge = expert_page;
    if (ssm_page) {
        const int64_t g = gcd64(expert_page, ssm_page);
        if (expert_page / g > INT64_MAX / ssm_page) return bad("pmoe_tiers_create: huge page too large");
        huge = expert_page / g * ssm_page;
    }
    pmoe_tiers* t = new pmoe_tiers;
    t->huge_bytes = huge;
    t->size[PMOE_PAGE_EXPERT] = expert_page;
    t->size[PMOE_PAGE_SSM] = ssm_page;
    t->size[PMOE_PAGE_KV] = kv_page;
    t->size[PMOE_PAGE_CONV] = conv_page;
    t->n_huge = pool_bytes / huge;
    t->huge.assign(t->n_huge, Huge{});
    for (int64_t h = 0; h < t->n_huge; ++h) t->free_huge.insert(h);
    *out = t;
    return PMOE_OK;
}

extern "C" pmoe_status pmoe_tiers_destroy(pmoe_tiers_t t) {
    delete t;
    return PMOE_OK;
}

extern "C" pmoe_status pmoe_tiers_alloc(pmoe_tiers_t t, int32_t kind, int64_t owner, int64_t* offset) {
    if (!t || !offset || kind < PMOE_PAGE_EXPERT || kind > PMOE_PAGE_CONV || owner < 0)
        return bad("pmoe_tiers_alloc: tiers and offset non-NULL, kind in range, owner >= 0");
    if (t->size[kind] == 0) return bad("pmoe_tiers_alloc: the pool has no pages of this kind");
    if (kind <= PMOE_PAGE_SSM) {
        *offset = take_mid(t, kind);
        if (*offset >= 0) t->live_mid[kind].insert(*offset);
    } else {
        *offset = take_small(t, kind, owner);
    }
    return PMOE_OK;
}

extern "C" pmoe_status pmoe_tiers_free(pmoe_tiers_t t, int32_t kind, int64_t offset) {
    if (!t || kind < PMOE_PAGE_EXPERT || kind > PMOE_PAGE_CONV)
        return bad("pmoe_tiers_free: tiers non-NULL, kind in range");
    if (kind <= PMOE_PAGE_SSM) {
        if (!t->live_mid[kind].count(offset)) return bad("pmoe_tiers_free: not a live page of this kind");
        t->live_mid[kind].erase(offset);
        give_mid(t, kind, offset);
        return PMOE_OK;
    }
    if (offset < 0) return bad("pmoe_tiers_free: not a live page of this kind");
    const int64_t e = offset - offset % t->size[PMOE_PAGE_EXPERT];
    auto it = t->split.find(e);
    if (it == t->split.end() || it->second.kind != kind)
        return bad("pmoe_tiers_free: not a live page of this kind");
    Split& sp = it->second;
    const int64_t slot = (offset - e) / t->size[kind];
    if ((offset - e) % t->size[kind] || sp.owner[slot] < 0)
        return bad("pmoe_tiers_free: not a live page of this kind");
    const int s = kind - PMOE_PAGE_KV;
    auto& pages = t->by_owner[s][sp.owner[slot]];
    if (--pages[e] == 0) pages.erase(e);
    if (pages.empty()) t->by_owner[s].erase(sp.owner[slot]);
    sp.owner[slot] = -1;
    sp.live -= 1;
    if (sp.live == 0) {                 // every small page back: an expert page again
        t->has_free[s].erase(e);
        t->split.erase(it);
        give_mid(t, PMOE_PAGE_EXPERT, e);
    } else {
        t->has_free[s].insert(e);
    }
    return PMOE_OK;
}

extern "C" pmoe_status pmoe_tiers_stats(pmoe_tiers_t t, int64_t* c) {
    if (!t || !c) return bad("pmoe_tiers_stats: NULL argument");
    int64_t free_small = 0;
    for (const auto& kv : t->split) free_small += (int64_t)kv.second.owner.size() - kv.second.live;
    c[0] = t->huge_bytes;
    c[1] = (int64_t)t->free_huge.size();
    c[2] = (int64_t)t->free_mid[0].size();
    c[3] = (int64_t)t->free_mid[1].size();
    c[4] = (int64_t)t->live_mid[0].size();
    c[5] = (int64_t)t->live_mid[1].size();
    c[6] = (int64_t)t->split.size();
    c[7] = free_small;
    return PMOE_OK;
}
