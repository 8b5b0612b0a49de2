// residency.cu -- host-side replacement policies for the expert slot pool and the
// driver that applies their decisions (moe_policy_* in moe.h). Host code only: no
// kernel lives here; moe_policy_apply enqueues through moe_slot_evict / moe_slot_load.
//
// kairos-engine README, "Decode, 2026-09-28/29" (an LRU cache of experts; resolving
// a layer stamps its slots most recently used so the layer cannot evict its own
// experts) and "2026-09-29: which experts to keep" (decayed frequency with a
// 32-token half-life and a 2-token recency guard); Strata article, "The cache's
// replacement rule" (per-layer float counters, swaps of the hottest missing against
// the coldest resident experts with a 1.5 hysteresis and a threshold of 2, at most
// 96 swaps per round, counters x 0.7 per round).
#include <algorithm>
#include <cmath>
#include <limits>
#include <queue>
#include <vector>

#include "moe_internal.cuh"

struct moe_policy {
    moe_policy_params pr;
    int L = 0, E = 0, n = 0;      // layers, experts, pairs
    std::vector<uint8_t> res;     // resident flag per pair
    std::vector<uint8_t> mark;    // pair is in the event being served
    int n_res = 0;
    std::vector<int> rlist, rpos;  // resident pairs (any order) and each pair's index in it
    // LRU order: doubly linked list of resident pairs, head = most recent
    std::vector<int> prev, next;
    int head = -1, tail = -1;
    // decayed frequency
    std::vector<double> score;
    std::vector<long long> tau, last;  // token of the score's last update / last access (-1: never)
    std::vector<unsigned long long> stamp;  // access order (0: never)
    unsigned long long clock = 0;
    double f = 1.0;  // score factor per token, 2^(-1 / half_life)
    std::vector<double> fpow;  // fpow[d] = pow(f, d), the factor after d tokens
    // Victim search without a scan. Every score decays by the same factor per token,
    // so log2(score) + tau / half_life orders the resident pairs as their decayed
    // scores do (up to rounding). Accessed resident pairs sit in a min-heap on that
    // key; never-accessed ones (score 0, the lowest of all) in a min-heap on the pair
    // index. Records carry the pair's version and go stale when it changes.
    struct Rec {
        double key;
        int k;
        unsigned v;
    };
    std::vector<Rec> heap;
    std::vector<std::pair<int, unsigned>> zheap;
    std::vector<unsigned> ver;
    // accessed pairs inside the recency guard wait here, on the token their guard
    // ends, and join the heap then: the heap holds unguarded pairs only
    struct Held {
        long long release;
        int k;
        unsigned v;
    };
    std::vector<Held> held;
    // LFU with swaps
    std::vector<float> cnt;
    long long token = 0;
};

namespace {

using moe::set_error;

void lru_unlink(moe_policy *p, int k) {
    if (p->prev[k] >= 0) p->next[p->prev[k]] = p->next[k];
    else p->head = p->next[k];
    if (p->next[k] >= 0) p->prev[p->next[k]] = p->prev[k];
    else p->tail = p->prev[k];
    p->prev[k] = p->next[k] = -1;
}

void lru_push_front(moe_policy *p, int k) {
    p->prev[k] = -1;
    p->next[k] = p->head;
    if (p->head >= 0) p->prev[p->head] = k;
    p->head = k;
    if (p->tail < 0) p->tail = k;
}

void lru_push_back(moe_policy *p, int k) {
    p->next[k] = -1;
    p->prev[k] = p->tail;
    if (p->tail >= 0) p->next[p->tail] = k;
    p->tail = k;
    if (p->head < 0) p->head = k;
}

void list_add(moe_policy *p, int k) {
    p->rpos[k] = (int)p->rlist.size();
    p->rlist.push_back(k);
}

void list_remove(moe_policy *p, int k) {
    const int i = p->rpos[k], last = p->rlist.back();
    p->rlist[i] = last;
    p->rpos[last] = i;
    p->rlist.pop_back();
    p->rpos[k] = -1;
}

struct RecAfter {  // heap order: lowest key (then lowest pair) on top
    bool operator()(const moe_policy::Rec &a, const moe_policy::Rec &b) const {
        return a.key > b.key || (a.key == b.key && a.k > b.k);
    }
};

void heap_push(moe_policy *p, const moe_policy::Rec &r) {
    p->heap.push_back(r);
    std::push_heap(p->heap.begin(), p->heap.end(), RecAfter());
}

void zheap_push(moe_policy *p, int k, unsigned v) {
    p->zheap.emplace_back(k, v);
    std::push_heap(p->zheap.begin(), p->zheap.end(), std::greater<std::pair<int, unsigned>>());
}

struct HeldAfter {  // earliest release on top
    bool operator()(const moe_policy::Held &a, const moe_policy::Held &b) const { return a.release > b.release; }
};

bool guarded_now(const moe_policy *p, int k) {
    return p->last[k] >= 0 && p->token - p->last[k] < p->pr.recency_guard;
}

double df_key(const moe_policy *p, int k) { return std::log2(p->score[k]) + (double)p->tau[k] / p->pr.half_life; }

// File resident pair k (version v) where it belongs now: held while inside the guard,
// else the heap (accessed) or the never-accessed heap.
void df_place(moe_policy *p, int k, unsigned v) {
    if (guarded_now(p, k)) {
        p->held.push_back({p->last[k] + p->pr.recency_guard, k, v});
        std::push_heap(p->held.begin(), p->held.end(), HeldAfter());
    } else if (p->score[k] > 0.0) {
        heap_push(p, {df_key(p, k), k, v});
    } else {
        zheap_push(p, k, v);
    }
}

// (Re)file resident pair k of the decayed-frequency policy after its score changed or
// it became resident; stale records are dropped when they reach the top, and the
// structures are rebuilt from the resident list when stale records pile up.
void df_file(moe_policy *p, int k) {
    if (p->pr.kind != MOE_POLICY_DECAYED_FREQ || !p->res[k]) return;
    df_place(p, k, ++p->ver[k]);
    if (p->heap.size() + p->zheap.size() + p->held.size() > 4 * (size_t)p->n_res + 256) {
        p->heap.clear();
        p->zheap.clear();
        p->held.clear();
        for (int r : p->rlist) df_place(p, r, p->ver[r]);
    }
}

// The token advanced: pairs whose guard has ended join the heap.
void df_release(moe_policy *p) {
    while (!p->held.empty() && p->held.front().release <= p->token) {
        const moe_policy::Held h = p->held.front();
        std::pop_heap(p->held.begin(), p->held.end(), HeldAfter());
        p->held.pop_back();
        if (h.v == p->ver[h.k] && p->res[h.k]) heap_push(p, {df_key(p, h.k), h.k, h.v});
    }
}

void make_resident(moe_policy *p, int k) {
    p->res[k] = 1;
    ++p->n_res;
    list_add(p, k);
    if (p->pr.kind == MOE_POLICY_LRU) lru_push_front(p, k);
    df_file(p, k);
}

void make_absent(moe_policy *p, int k) {
    p->res[k] = 0;
    --p->n_res;
    list_remove(p, k);
    if (p->pr.kind == MOE_POLICY_LRU) lru_unlink(p, k);
    ++p->ver[k];
}

// pow(f, d) for d tokens, the same value a direct pow call gives
double fpow(moe_policy *p, long long d) {
    while ((long long)p->fpow.size() <= d) p->fpow.push_back(std::pow(p->f, (double)p->fpow.size()));
    return p->fpow[d];
}

double decayed(moe_policy *p, int k) { return p->score[k] * fpow(p, p->token - p->tau[k]); }

// The decayed-frequency order: lower decayed score; equal scores to the least
// recently used, then the lower pair.
bool df_before(moe_policy *p, int k, double s, int best, double bs) {
    return best < 0 || s < bs || (s == bs && (p->stamp[k] < p->stamp[best] || (p->stamp[k] == p->stamp[best] && k < best)));
}

int scan_victim(moe_policy *p);

// Decayed-frequency victim from the heaps. A never-accessed pair (score 0) comes first.
// Otherwise the lowest key among eligible pairs, and every eligible pair whose key is
// within a slack far above rounding of it, are compared exactly as the scan compares
// them (decayed score, recency, pair): a pair beyond the slack has a decayed score
// larger by a factor of at least 2^slack, which rounding cannot undo. Scores that
// underflow go to the scan.
int heap_victim(moe_policy *p) {
    {
        std::vector<std::pair<int, unsigned>> back;
        int victim = -1;
        auto zafter = std::greater<std::pair<int, unsigned>>();
        while (!p->zheap.empty()) {
            const std::pair<int, unsigned> r = p->zheap.front();
            const int k = r.first;
            std::pop_heap(p->zheap.begin(), p->zheap.end(), zafter);
            p->zheap.pop_back();
            if (r.second != p->ver[k] || !p->res[k]) continue;  // stale
            back.push_back(r);
            if (p->mark[k]) continue;
            victim = k;
            break;
        }
        for (const auto &r : back) zheap_push(p, r.first, r.second);
        if (victim >= 0) return victim;
    }
    // unguarded accessed pairs: the heap holds exactly these (held pairs join it when
    // their guard ends), so the event's own pairs are the only ones passed over
    constexpr double kSlack = 1e-6;  // in log2 units: a factor of 1 + 6.9e-7
    constexpr int kMaxSkip = 64;     // more passed-over pairs than this: the scan is cheaper
    std::vector<moe_policy::Rec> back;
    int best = -1, skipped = 0;
    double bs = 0.0, k0 = 0.0;
    bool have = false, scan = false;
    while (!p->heap.empty()) {
        const moe_policy::Rec r = p->heap.front();
        if (have && r.key > k0 + kSlack * (1.0 + std::fabs(k0))) break;
        std::pop_heap(p->heap.begin(), p->heap.end(), RecAfter());
        p->heap.pop_back();
        const int k = r.k;
        if (r.v != p->ver[k] || !p->res[k]) continue;  // stale
        back.push_back(r);
        if (p->mark[k] || guarded_now(p, k)) {
            if (++skipped > kMaxSkip) {
                scan = true;
                break;
            }
            continue;
        }
        if (!have) {
            have = true;
            k0 = r.key;
        }
        const double s = decayed(p, k);
        if (df_before(p, k, s, best, bs)) {
            best = k;
            bs = s;
        }
    }
    for (const auto &r : back) heap_push(p, r);
    if (!scan && best >= 0 && bs >= std::numeric_limits<double>::min()) return best;
    // underflowed scores, or every pair outside the event inside the guard (then the
    // guarded ones compete): the scan decides
    return scan_victim(p);
}

// Victim for a load, or -1: never a pair of the event being served.
int pick_victim(moe_policy *p) {
    if (p->pr.kind == MOE_POLICY_LRU) {
        for (int k = p->tail; k >= 0; k = p->prev[k])
            if (!p->mark[k]) return k;
        return -1;
    }
    return heap_victim(p);
}

// The decayed-frequency victim by a scan of the resident pairs: lowest decayed score
// first among entries outside the recency guard, then among all.
int scan_victim(moe_policy *p) {
    for (int guarded = 1; guarded >= 0; --guarded) {
        int best = -1;
        double bs = 0.0;
        for (int k : p->rlist) {
            if (p->mark[k] || (guarded && guarded_now(p, k))) continue;
            const double s = decayed(p, k);
            if (df_before(p, k, s, best, bs)) {
                best = k;
                bs = s;
            }
        }
        if (best >= 0) return best;
    }
    return -1;
}

// One routing event (arguments checked by the caller): hits, then for the demand
// policies the loads with their victims, appended at the given plan pointers
// (load_layer may be NULL); returns the number of loads.
int route_event(moe_policy *p, int layer, const int32_t *ids, int n, uint8_t *hit, int32_t *load_layer,
                int32_t *load_expert, int32_t *evict_layer, int32_t *evict_expert) {
    // the event's distinct pairs, in event order
    std::vector<int> ev;
    ev.reserve(n);
    for (int i = 0; i < n; ++i) {
        const int k = layer * p->E + ids[i];
        if (hit) hit[i] = p->res[k];
        if (p->mark[k]) continue;
        p->mark[k] = 1;
        ev.push_back(k);
    }
    int nl = 0;
    if (p->pr.kind == MOE_POLICY_LFU_SWAP) {
        for (int k : ev) p->cnt[k] += 1.0f;
    } else {
        for (int k : ev) {
            if (p->pr.kind == MOE_POLICY_LRU) {
                if (p->res[k]) {
                    lru_unlink(p, k);
                    lru_push_front(p, k);
                }
            } else {
                p->score[k] = p->score[k] * fpow(p, p->token - p->tau[k]) + 1.0;
                p->tau[k] = p->token;
                p->last[k] = p->token;
                p->stamp[k] = ++p->clock;
                df_file(p, k);
            }
        }
        for (int k : ev) {
            if (p->res[k]) continue;
            int victim = -1;
            if (p->n_res >= p->pr.capacity) {
                victim = pick_victim(p);
                if (victim < 0) continue;  // the pool holds only this event's experts
                make_absent(p, victim);
            }
            make_resident(p, k);
            if (load_layer) load_layer[nl] = layer;
            load_expert[nl] = k % p->E;
            evict_layer[nl] = victim < 0 ? -1 : victim / p->E;
            evict_expert[nl] = victim < 0 ? -1 : victim % p->E;
            ++nl;
        }
    }
    for (int k : ev) p->mark[k] = 0;
    return nl;
}

}  // namespace

extern "C" {

MOE_API int moe_policy_create(const moe_policy_params *params, int n_layers, int n_experts, moe_policy **out) {
    if (!params || !out) return set_error(MOE_ERR_ARG, "null argument");
    const moe_policy_params &q = *params;
    if (q.kind < MOE_POLICY_LRU || q.kind > MOE_POLICY_LFU_SWAP) return set_error(MOE_ERR_ARG, "unknown policy %d", q.kind);
    if (n_layers < 1 || n_experts < 1 || (long long)n_layers * n_experts > (1LL << 26))
        return set_error(MOE_ERR_SHAPE, "n_layers=%d n_experts=%d", n_layers, n_experts);
    if (q.capacity < 1) return set_error(MOE_ERR_ARG, "capacity %d < 1", q.capacity);
    if (q.kind == MOE_POLICY_DECAYED_FREQ && !(q.half_life > 0.0))
        return set_error(MOE_ERR_ARG, "half_life must be positive");
    if (q.kind == MOE_POLICY_DECAYED_FREQ && q.recency_guard < 0) return set_error(MOE_ERR_ARG, "recency_guard < 0");
    if (q.kind == MOE_POLICY_LFU_SWAP && (q.swap_every < 1 || q.max_swaps < 0))
        return set_error(MOE_ERR_ARG, "swap_every %d / max_swaps %d", q.swap_every, q.max_swaps);
    moe_policy *p = new moe_policy;
    p->pr = q;
    p->L = n_layers;
    p->E = n_experts;
    p->n = n_layers * n_experts;
    p->res.assign(p->n, 0);
    p->mark.assign(p->n, 0);
    p->prev.assign(p->n, -1);
    p->next.assign(p->n, -1);
    p->score.assign(p->n, 0.0);
    p->tau.assign(p->n, 0);
    p->last.assign(p->n, -1);
    p->stamp.assign(p->n, 0);
    p->cnt.assign(p->n, 0.f);
    p->rpos.assign(p->n, -1);
    p->ver.assign(p->n, 0);
    p->rlist.reserve(q.capacity);
    if (q.kind == MOE_POLICY_DECAYED_FREQ) p->f = std::pow(2.0, -1.0 / q.half_life);
    *out = p;
    return MOE_OK;
}

MOE_API int moe_policy_destroy(moe_policy *p) {
    delete p;
    return MOE_OK;
}

MOE_API int moe_policy_seed(moe_policy *p, const int32_t *layers, const int32_t *experts, int n, int *n_placed) {
    if (!p || (n > 0 && (!layers || !experts))) return set_error(MOE_ERR_ARG, "null argument");
    // every pair is checked before any is placed: a bad list changes nothing
    for (int i = 0; i < n; ++i)
        if (layers[i] < 0 || layers[i] >= p->L || experts[i] < 0 || experts[i] >= p->E)
            return set_error(MOE_ERR_ARG, "pair (%d, %d) out of range", layers[i], experts[i]);
    int placed = 0;
    for (int i = 0; i < n && p->n_res < p->pr.capacity; ++i) {
        const int k = layers[i] * p->E + experts[i];
        if (p->res[k]) continue;
        // a profile lists the hottest first: seeded entries are older than any access,
        // the first listed the most recent of them
        p->res[k] = 1;
        ++p->n_res;
        list_add(p, k);
        if (p->pr.kind == MOE_POLICY_LRU) lru_push_back(p, k);
        df_file(p, k);
        ++placed;
    }
    if (n_placed) *n_placed = placed;
    return MOE_OK;
}

MOE_API int moe_policy_route(moe_policy *p, int layer, const int32_t *ids, int n, uint8_t *hit, int32_t *load_expert,
                             int32_t *evict_layer, int32_t *evict_expert, int *n_loads) {
    if (!p || (n > 0 && !ids)) return set_error(MOE_ERR_ARG, "null argument");
    if (layer < 0 || layer >= p->L) return set_error(MOE_ERR_ARG, "layer %d out of range", layer);
    for (int i = 0; i < n; ++i)
        if (ids[i] < 0 || ids[i] >= p->E) return set_error(MOE_ERR_ARG, "expert %d out of range", ids[i]);
    const bool demand = p->pr.kind != MOE_POLICY_LFU_SWAP;
    if (demand && (!load_expert || !evict_layer || !evict_expert || !n_loads))
        return set_error(MOE_ERR_ARG, "null plan buffers");
    const int nl = route_event(p, layer, ids, n, hit, nullptr, load_expert, evict_layer, evict_expert);
    if (n_loads) *n_loads = nl;
    return MOE_OK;
}

MOE_API int moe_policy_route_token(moe_policy *p, const int32_t *ids, int n_layers, int K, uint8_t *hit,
                                   int32_t *load_layer, int32_t *load_expert, int32_t *evict_layer,
                                   int32_t *evict_expert, int cap, int *n_loads) {
    if (!p || n_layers < 0 || K < 0 || ((long long)n_layers * K > 0 && !ids))
        return set_error(MOE_ERR_ARG, "null argument or negative size");
    if (n_layers > p->L) return set_error(MOE_ERR_ARG, "%d layers routed, the policy has %d", n_layers, p->L);
    const long long total = (long long)n_layers * K;
    for (long long i = 0; i < total; ++i)
        if (ids[i] < 0 || ids[i] >= p->E) return set_error(MOE_ERR_ARG, "expert %d out of range", ids[i]);
    const bool demand = p->pr.kind != MOE_POLICY_LFU_SWAP;
    if (demand && (!load_layer || !load_expert || !evict_layer || !evict_expert || !n_loads))
        return set_error(MOE_ERR_ARG, "null plan buffers");
    if (demand && cap < total) return set_error(MOE_ERR_ARG, "cap %d < n_layers * K = %lld", cap, total);
    int nl = 0;
    for (int l = 0; l < n_layers; ++l)
        nl += route_event(p, l, ids + (size_t)l * K, K, hit ? hit + (size_t)l * K : nullptr,
                          demand ? load_layer + nl : nullptr, demand ? load_expert + nl : nullptr,
                          demand ? evict_layer + nl : nullptr, demand ? evict_expert + nl : nullptr);
    if (n_loads) *n_loads = nl;
    return MOE_OK;
}

MOE_API int moe_policy_end_token(moe_policy *p, int32_t *load_layer, int32_t *load_expert, int32_t *evict_layer,
                                 int32_t *evict_expert, int cap, int *n_swaps) {
    if (!p) return set_error(MOE_ERR_ARG, "null argument");
    int ns = 0;
    ++p->token;
    if (p->pr.kind == MOE_POLICY_DECAYED_FREQ) df_release(p);
    if (p->pr.kind == MOE_POLICY_LFU_SWAP) {
        if (p->token % p->pr.swap_every == 0) {
            struct Swap {
                float gain;
                int layer, in, out;
            };
            std::vector<Swap> sw;
            std::vector<std::pair<float, int>> cand, vict;
            for (int l = 0; l < p->L; ++l) {
                cand.clear();
                vict.clear();
                for (int e = 0; e < p->E; ++e) {
                    const int k = l * p->E + e;
                    if (p->res[k]) vict.emplace_back(p->cnt[k], e);
                    else if (p->cnt[k] >= p->pr.min_count) cand.emplace_back(p->cnt[k], e);
                }
                std::sort(cand.begin(), cand.end(), [](const std::pair<float, int> &a, const std::pair<float, int> &b) {
                    return a.first != b.first ? a.first > b.first : a.second < b.second;
                });
                std::sort(vict.begin(), vict.end(), [](const std::pair<float, int> &a, const std::pair<float, int> &b) {
                    return a.first != b.first ? a.first < b.first : a.second < b.second;
                });
                const size_t m = std::min(cand.size(), vict.size());
                for (size_t i = 0; i < m; ++i) {
                    if (cand[i].first < vict[i].first + p->pr.margin) break;
                    sw.push_back(Swap{cand[i].first - vict[i].first, l, cand[i].second, vict[i].second});
                }
            }
            std::stable_sort(sw.begin(), sw.end(), [](const Swap &a, const Swap &b) { return a.gain > b.gain; });
            // with plan buffers, no more swaps than they hold (every swap made is reported)
            const bool out = load_layer && load_expert && evict_layer && evict_expert;
            size_t take = std::min(sw.size(), (size_t)p->pr.max_swaps);
            if (out) take = std::min(take, (size_t)(cap > 0 ? cap : 0));
            for (size_t i = 0; i < take; ++i) {
                const Swap &s = sw[i];
                make_absent(p, s.layer * p->E + s.out);
                make_resident(p, s.layer * p->E + s.in);
                if (out) {
                    load_layer[i] = s.layer;
                    load_expert[i] = s.in;
                    evict_layer[i] = s.layer;
                    evict_expert[i] = s.out;
                }
            }
            ns = (int)take;
        }
        for (float &c : p->cnt) c *= p->pr.decay;
    }
    if (n_swaps) *n_swaps = ns;
    return MOE_OK;
}

MOE_API int moe_policy_resident(const moe_policy *p, int layer, int expert, int *resident) {
    if (!p || !resident) return set_error(MOE_ERR_ARG, "null argument");
    if (layer < 0 || layer >= p->L || expert < 0 || expert >= p->E) return set_error(MOE_ERR_ARG, "pair out of range");
    *resident = p->res[layer * p->E + expert];
    return MOE_OK;
}

MOE_API int moe_policy_count(const moe_policy *p, int *n_resident) {
    if (!p || !n_resident) return set_error(MOE_ERR_ARG, "null argument");
    *n_resident = p->n_res;
    return MOE_OK;
}

MOE_API int moe_policy_belady(const int32_t *ids, int T, int n_layers, int K, int n_experts, int capacity,
                              const int32_t *seed_layers, const int32_t *seed_experts, int n_seed, long long *hits) {
    if (!hits || (T > 0 && !ids) || (n_seed > 0 && (!seed_layers || !seed_experts)))
        return set_error(MOE_ERR_ARG, "null argument");
    if (T < 0 || n_layers < 1 || K < 1 || n_experts < 1 || capacity < 1 ||
        (long long)n_layers * n_experts > (1LL << 26))
        return set_error(MOE_ERR_SHAPE, "T=%d n_layers=%d K=%d n_experts=%d capacity=%d", T, n_layers, K, n_experts,
                         capacity);
    const long long never = std::numeric_limits<long long>::max();
    // the events' distinct pairs in order, and each position's next use
    std::vector<int> seq;
    std::vector<long long> ev_end;  // end position of each event
    seq.reserve((size_t)T * n_layers * K);
    std::vector<int> mark((size_t)n_layers * n_experts, -1);
    long long ev = 0;
    for (int t = 0; t < T; ++t)
        for (int l = 0; l < n_layers; ++l, ++ev) {
            for (int k = 0; k < K; ++k) {
                const int e = ids[((size_t)t * n_layers + l) * K + k];
                if (e < 0 || e >= n_experts) return set_error(MOE_ERR_ARG, "expert %d out of range", e);
                const int key = l * n_experts + e;
                if (mark[key] == ev) continue;
                mark[key] = (int)ev;
                seq.push_back(key);
            }
            ev_end.push_back((long long)seq.size());
        }
    const size_t n = seq.size();
    std::vector<long long> nxt(n), next_use((size_t)n_layers * n_experts, never);
    for (size_t i = n; i-- > 0;) {
        nxt[i] = next_use[seq[i]];
        next_use[seq[i]] = (long long)i;
    }
    // next_use now holds each pair's first use
    std::vector<uint8_t> res((size_t)n_layers * n_experts, 0), in_ev((size_t)n_layers * n_experts, 0);
    std::priority_queue<std::pair<long long, int>> heap;  // (next use, pair), farthest first
    int n_res = 0;
    for (int i = 0; i < n_seed && n_res < capacity; ++i) {
        const int l = seed_layers[i], e = seed_experts[i];
        if (l < 0 || l >= n_layers || e < 0 || e >= n_experts) return set_error(MOE_ERR_ARG, "seed pair out of range");
        const int key = l * n_experts + e;
        if (res[key]) continue;
        res[key] = 1;
        ++n_res;
        heap.push({next_use[key], key});
    }
    long long h = 0;
    size_t pos = 0;
    std::vector<std::pair<long long, int>> skipped;
    for (long long end : ev_end) {
        const size_t b = pos;
        for (size_t i = b; i < (size_t)end; ++i) in_ev[seq[i]] = 1;
        for (size_t i = b; i < (size_t)end; ++i) {
            const int key = seq[i];
            if (res[key]) {
                ++h;
                next_use[key] = nxt[i];
                heap.push({nxt[i], key});
            }
        }
        for (size_t i = b; i < (size_t)end; ++i) {
            const int key = seq[i];
            if (res[key]) continue;
            if (n_res >= capacity) {
                int victim = -1;
                skipped.clear();
                while (!heap.empty()) {
                    const std::pair<long long, int> top = heap.top();
                    heap.pop();
                    if (!res[top.second] || next_use[top.second] != top.first) continue;  // stale
                    if (in_ev[top.second]) {
                        skipped.push_back(top);
                        continue;
                    }
                    victim = top.second;
                    break;
                }
                for (const auto &sk : skipped) heap.push(sk);
                if (victim < 0) continue;
                res[victim] = 0;
                --n_res;
            }
            res[key] = 1;
            ++n_res;
            next_use[key] = nxt[i];
            heap.push({nxt[i], key});
        }
        for (size_t i = b; i < (size_t)end; ++i) in_ev[seq[i]] = 0;
        pos = (size_t)end;
    }
    *hits = h;
    return MOE_OK;
}

MOE_API int moe_policy_apply(moe_slots *slots, int n_experts, const void *const *blobs, size_t nbytes,
                             const int32_t *load_layer, const int32_t *load_expert, const int32_t *evict_layer,
                             const int32_t *evict_expert, int n, moe_stream_t stream) {
    if (!slots || (n > 0 && (!blobs || !load_layer || !load_expert || !evict_layer || !evict_expert)))
        return set_error(MOE_ERR_ARG, "null argument");
    for (int i = 0; i < n; ++i) {
        if (evict_layer[i] >= 0) {
            const int rc = moe_slot_evict(slots, evict_layer[i], evict_expert[i], stream);
            if (rc) return rc;
        }
        if (load_layer[i] < 0 || load_expert[i] < 0 || load_expert[i] >= n_experts)
            return set_error(MOE_ERR_ARG, "load pair (%d, %d) out of range", load_layer[i], load_expert[i]);
        const void *blob = blobs[(size_t)load_layer[i] * n_experts + load_expert[i]];
        if (!blob) return set_error(MOE_ERR_ARG, "no blob for (%d, %d)", load_layer[i], load_expert[i]);
        const int rc = moe_slot_load(slots, load_layer[i], load_expert[i], blob, nbytes, stream);
        if (rc) return rc;
    }
    return MOE_OK;
}

}  // extern "C"
