// pst_plan_create: KV-guided grouping, mask packing, cost model and the
// partitioner that chooses the KV-axis split b_k of every node.
//
// CoDec, "workload balancing": each node is a task T[i] = (n_q[i], n[i]); the
// query axis is never split (b_q = 1) and the KV axis is split b_k[i] ways; the
// objective is the smallest maximum per-block cost over assignments A of the
// sub-tasks to m blocks. A binary search finds the lower bound cost_l on the
// block cost (the average block cost rises monotonically as splits get finer),
// b_k[i] is bounded by ceil(C_est(n_q[i], n[i]) / cost_l), and a search over
// the b_k picks the split with the best list schedule (Graham 1966).
//
// DEFT, Algorithm 1 (QKV preparation): QMapKV (per query its prefix nodes) and
// KVMapQ (per node the queries sharing it). DEFT's bit causal mask: one 64-bit
// word per query records which tokens of a chunk it may see.
#include <algorithm>
#include <cstdint>
#include <chrono>
#include <memory>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <numeric>
#include <queue>
#include <unordered_map>
#include <string>

#include "pst_internal.h"

namespace pst {

int device_sm_count(int* out);  // attn.cu

// ------------------------------------------------------------------ cost model
// Profile-based estimator C_est(rows, tokens) (CoDec "profile-based cost
// estimation"): a measured table per PAC kind (CUDA core, tensor core with P
// rounded once, tensor core with exact P), bilinear in (log rows, log tokens)
// and linear in tokens past the last grid point. The tables measured on a
// GB300 are built in; an analytic model stands in for shapes they do not
// cover (d != 128, fp32, the mma.sync engine).
namespace {
struct CostTable {
    bool set = false;
    std::vector<double> lr, ln, us;  // log rows, log tokens, values [n_r][n_n]
};
std::mutex g_cost_mu;
CostTable g_cost[kCostKinds];

// The built-in tables (written by the package's cost_fit.py).
#include "cost_table_gb300.inc"

CostTable builtin_table(int k) {
    CostTable T;
    const BuiltinCostTable& b = kBuiltinCost[k];
    if (b.n_r == 0) return T;
    for (int i = 0; i < b.n_r; ++i) T.lr.push_back(std::log(b.rows[i]));
    for (int j = 0; j < b.n_n; ++j) T.ln.push_back(std::log(b.tokens[j]));
    T.us.assign(b.us, b.us + b.n_r * b.n_n);
    T.set = true;
    return T;
}

struct BuiltinInstaller {
    BuiltinInstaller() {
        for (int k = 0; k < kCostKinds; ++k) g_cost[k] = builtin_table(k);
    }
} g_builtin_installer;

double interp(const std::vector<double>& g, double x, int* i0) {
    // returns the fractional position of x between g[i0] and g[i0+1], clamped
    int n = (int)g.size();
    if (n == 1 || x <= g[0]) { *i0 = 0; return 0.0; }
    if (x >= g[n - 1]) { *i0 = std::max(0, n - 2); return n == 1 ? 0.0 : 1.0; }
    int i = (int)(std::upper_bound(g.begin(), g.end(), x) - g.begin()) - 1;
    *i0 = i;
    return (x - g[i]) / (g[i + 1] - g[i]);
}
}  // namespace

// Analytic stand-in, per PAC thread block with every SM busy: a fixed block
// cost plus the larger of its HBM time and its arithmetic time, plus the
// partial output it writes and POR reads back.
static double analytic_cost(int kind, double rows, double tokens, double bytes_per_tok, int d,
                            int num_sms) {
    const double bw_sm = 6.0e6 / std::max(1, num_sms);        // bytes per us per SM
    const double t0 = 1.5;                                     // us per block
    // a thin-PAC item covers kThinHeads kv heads
    const double heads = kind == 3 ? kThinHeads : 1;
    const double mem = tokens * bytes_per_tok * heads / bw_sm;
    double cmp;
    if (kind == 3) {
        // tcgen05 thin PAC: one block per SM streams its 32 KB tiles at the SM's
        // share of HBM; the small MMAs and the softmax stay below that
        cmp = 0.0;
    } else if (kind == 1) {
        // tcgen05 (measured on GB300): a 64-token tile costs ~3300 clk with
        // two 128-row halves (S = Q K^T and the hi and lo PV products share
        // the tensor pipe and tensor memory with the softmax's loads and
        // stores) and ~1000 clk with one half split over the two softmax
        // groups; ~2 GHz
        const double per_tok = rows > 128 ? 52.0 : 16.0;
        const double t_mma = tokens * per_tok * (d / 128.0) / 2000.0;
        const double t_sfu = tokens * rows / (16.0 * 2000.0);
        cmp = std::max(t_mma, t_sfu);
    } else {
        const double instr = 8.0 + 11.0 * rows;                // warp instructions per token
        cmp = tokens * instr * (d / 128.0) / (4.0 * 1800.0);   // 4 issue/clk at 1.8 GHz
    }
    const double part = heads * rows * (4.0 * d + 4.0) * 2.0 / bw_sm;
    return t0 + std::max(mem, cmp) + part;
}

double cost_estimate(int kind, double rows, double tokens) {
    return analytic_cost(kind == 3 ? 3 : kind ? 1 : 0, rows, tokens, 512.0, 128, 152);
}

// kind: 0 CUDA core, 1 tensor core (P rounded once), 2 tensor core (exact P),
// 3 tcgen05 thin PAC
static double cost_us(int kind, double rows, double tokens, double bytes_per_tok, int d,
                      int num_sms) {
    {
        std::lock_guard<std::mutex> lk(g_cost_mu);
        const CostTable& T = g_cost[kind];
        if (T.set && d == 128 && bytes_per_tok == 512.0) {
            const double t_max = std::exp(T.ln.back());
            const double scale = tokens > t_max ? tokens / t_max : 1.0;   // linear past the grid
            int i, j;
            double fr = interp(T.lr, std::log(std::max(1.0, rows)), &i);
            double ft = interp(T.ln, std::log(std::max(1.0, std::min(tokens, t_max))), &j);
            const int nn = (int)T.ln.size();
            auto at = [&](int a, int b) {
                a = std::min(a, (int)T.lr.size() - 1);
                b = std::min(b, nn - 1);
                return T.us[(size_t)a * nn + b];
            };
            double v0 = at(i, j) * (1 - ft) + at(i, j + 1) * ft;
            double v1 = at(i + 1, j) * (1 - ft) + at(i + 1, j + 1) * ft;
            return (v0 * (1 - fr) + v1 * fr) * scale;
        }
    }
    return analytic_cost(kind == 3 ? 3 : kind ? 1 : 0, rows, tokens, bytes_per_tok, d, num_sms);
}

}  // namespace pst

using namespace pst;

extern "C" int pst_cost_set_table(int32_t kind, int32_t n_r, const float* rows, int32_t n_n,
                                  const float* tokens, const float* us) {
    if (kind < 0 || kind >= kCostKinds) return fail(PST_EINVAL, "cost_set_table: kind must be 0, 1, 2 or 3");
    std::lock_guard<std::mutex> lk(g_cost_mu);
    CostTable& T = g_cost[kind];
    if (n_r < 0) {
        T = builtin_table(kind);  // back to the built-in table
        return PST_OK;
    }
    if (n_r == 0 || n_n <= 0 || !rows || !tokens || !us) {
        T = CostTable();  // the analytic model
        return PST_OK;
    }
    CostTable nt;
    for (int i = 0; i < n_r; ++i) {
        if (rows[i] <= 0 || (i && rows[i] <= rows[i - 1]))
            return fail(PST_EINVAL, "cost_set_table: rows must be positive and increasing");
        nt.lr.push_back(std::log((double)rows[i]));
    }
    for (int j = 0; j < n_n; ++j) {
        if (tokens[j] <= 0 || (j && tokens[j] <= tokens[j - 1]))
            return fail(PST_EINVAL, "cost_set_table: tokens must be positive and increasing");
        nt.ln.push_back(std::log((double)tokens[j]));
    }
    nt.us.assign(us, us + (size_t)n_r * n_n);
    nt.set = true;
    T = std::move(nt);
    return PST_OK;
}

extern "C" double pst_cost_estimate(int32_t kind, double rows, double tokens) {
    if (kind < 0 || kind >= kCostKinds) return -1.0;
    return cost_us(kind, rows, tokens, 512.0, 128, 152);
}

extern "C" void pst_plan_opts_default(pst_plan_opts* o) {
    if (!o) return;
    o->split_policy = PST_SPLIT_COST_MODEL;
    o->fixed_chunk = 1024;
    o->tc_min_rows = 16;
    o->pack_masks = 1;
    o->num_sms = 0;
    o->slots_per_sm = 1;
    o->tc_engine = 0;
    o->tc_block_rows = 256;
    o->p_bf16_min_tokens = kPBf16MinTokens;
    o->thin_engine = 0;
    o->debug_stall = 0;
    o->side_streams = 0;
    o->flatten_candidates = 0;
}

namespace {

int64_t align256(int64_t x) { return (x + 255) & ~int64_t(255); }

// Chunk boundaries of a node: the node's page-space span [fo, fo+len) is cut
// at multiples of the kernel's tile size (`blk` tokens) so that every chunk
// starts on a TMA tile.
struct Span {
    int32_t fo, len, first_block, n_blocks, blk;
};
Span node_span(int32_t fo, int32_t len, int32_t blk) {
    Span s{fo, len, fo / blk, 0, blk};
    const int32_t end_block = (fo + len + blk - 1) / blk;
    s.n_blocks = std::max(1, end_block - s.first_block);
    return s;
}
// token range [b, e) of chunk k of b_k
void chunk_range(const Span& s, int32_t bk, int32_t k, int32_t* b, int32_t* e) {
    const int64_t blk0 = s.first_block + (int64_t)s.n_blocks * k / bk;
    const int64_t blk1 = s.first_block + (int64_t)s.n_blocks * (k + 1) / bk;
    int64_t p0 = std::max<int64_t>(blk0 * s.blk, s.fo);
    int64_t p1 = std::min<int64_t>(blk1 * s.blk, (int64_t)s.fo + s.len);
    *b = (int32_t)(p0 - s.fo);
    *e = (int32_t)std::max<int64_t>(p1 - s.fo, p0 - s.fo);
}

// KV tokens per pipeline tile of the kernel that runs a task of `kind`
// (`thin`: thin chunks run on the tcgen05 thin PAC, one 16-row box per tile).
int32_t tile_tokens(int kind, const pst_plan_opts& o, bool thin) {
    if (kind == 1) return o.tc_engine == 0 ? kTcTileTokens : kTileTokens;
    return thin ? kBoxRows : kTileTokens;
}

// Rows per head of a thin-PAC item: 4 when the chunk has at most 4, else 8.
int32_t thin_rows(int32_t rows) { return rows <= 4 ? 4 : kThinRows; }

int32_t cc_row_tile(int32_t rows) {
    if (rows <= 1) return 1;
    if (rows <= 2) return 2;
    if (rows <= 4) return 4;
    return 8;
}

struct ItemCost {
    double cost;
    int32_t chunk;
    int16_t head, rb;
    int8_t klass;   // launch: 0 tensor core, 1 tensor core exact P, 2 + k CUDA core row tile 8 >> k
};

// Graham list scheduling (largest first) of item costs onto m slots: sorts
// v into that order and returns the makespan; slot (nullable) receives, per
// position of the sorted v, the slot the item went to (the least-loaded one,
// the lowest index among equals).
double list_schedule(std::vector<ItemCost>& v, int m, std::vector<int>* slot = nullptr) {
    std::sort(v.begin(), v.end(), [](const ItemCost& a, const ItemCost& b) {
        if (a.cost != b.cost) return a.cost > b.cost;
        if (a.chunk != b.chunk) return a.chunk < b.chunk;
        if (a.head != b.head) return a.head < b.head;
        return a.rb < b.rb;
    });
    using Slot = std::pair<double, int>;
    std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> pq;
    for (int i = 0; i < m; ++i) pq.push({0.0, i});
    if (slot) slot->assign(v.size(), 0);
    double mk = 0;
    for (size_t k = 0; k < v.size(); ++k) {
        Slot s = pq.top();
        pq.pop();
        s.first += v[k].cost;
        mk = std::max(mk, s.first);
        if (slot) (*slot)[k] = s.second;
        pq.push(s);
    }
    return mk;
}

// `n` items of one launch class and one cost (a chunk's row block over the
// kv heads). Which of several equal-cost items goes first does not change
// any SM's load, so the dispatcher's view below depends only on the
// multiset of (class, cost) and takes the items as such runs.
struct CostRun {
    double cost;
    int32_t n;
    int8_t klass;   // as ItemCost::klass
};

// The block dispatcher's view of one decode call, used to score a partition:
// the tensor-core launches come first and hold an SM per block (largest
// first, the exact-P launch after the other); the CUDA-core launches run one
// after the other on their own stream with `cc_per_sm[k]` blocks per SM, a
// block taking cc_per_sm[k] x C_est of wall time (C_est is per-SM-slot
// throughput), on the SMs the tensor-core blocks leave and, once those
// retire, on theirs. Sorts v; returns the time the last block ends.
double simulate_call(std::vector<CostRun>& v, int num_sms, const int (&cc_per_sm)[4]) {
    std::sort(v.begin(), v.end(), [](const CostRun& a, const CostRun& b) {
        if (a.klass != b.klass) return a.klass < b.klass;
        return a.cost > b.cost;
    });
    using Slot = std::pair<double, int>;
    std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> sm;
    for (int i = 0; i < num_sms; ++i) sm.push({0.0, i});
    std::vector<double> sm_free(num_sms, 0.0);
    size_t i = 0;
    double end = 0;
    for (; i < v.size() && v[i].klass < 2; ++i) {
        for (int32_t r = 0; r < v[i].n; ++r) {
            Slot x = sm.top();
            sm.pop();
            x.first += v[i].cost;
            sm_free[x.second] = x.first;
            end = std::max(end, x.first);
            sm.push(x);
        }
    }
    double start = 0;   // a CUDA-core launch starts when the previous one has ended
    while (i < v.size()) {
        const int k = v[i].klass - 2;
        const int per = std::max(1, cc_per_sm[k]);
        std::priority_queue<double, std::vector<double>, std::greater<double>> slots;
        for (int s2 = 0; s2 < num_sms; ++s2)
            for (int b = 0; b < per; ++b) slots.push(std::max(start, sm_free[s2]));
        double cls_end = start;
        for (; i < v.size() && v[i].klass - 2 == k; ++i) {
            for (int32_t r = 0; r < v[i].n; ++r) {
                double t = slots.top();
                slots.pop();
                t += per * v[i].cost;
                cls_end = std::max(cls_end, t);
                slots.push(t);
            }
        }
        start = cls_end;
        end = std::max(end, cls_end);
    }
    return end;
}

}  // namespace

namespace pst {
// CUDA-core PAC blocks that fit on one SM for a row tile (pac_cc.cu); -1 if
// no device can be asked.
int cc_blocks_per_sm(pst_dtype dt, int d, int r_tile);
}  // namespace pst

struct Planner {
    const Tree& T;
    pst_plan& P;
    int num_sms = 152;
    double bytes_per_tok = 0;
    int cc_per_sm[4] = {1, 3, 3, 3};   // row tiles 8, 4, 2, 1 (the thin PAC: class 0, one per SM)

    Planner(const Tree& t, pst_plan& p) : T(t), P(p) {}

    // cost kind of a task: 0 CUDA core, 1 tensor core with P rounded once,
    // 2 tensor core with exact P (a node shorter than p_bf16_min_tokens)
    int cost_kind(const Task& t) const {
        if (t.kind == 0) return P.thin ? 3 : 0;
        const int32_t p_single = P.opts.p_bf16_min_tokens < 0 ? INT32_MAX : P.opts.p_bf16_min_tokens;
        return t.n_tok < p_single ? 2 : 1;
    }

    double item_cost(const Task& t, int rows_blk, int tokens) const {
        if (t.kind == 1 && P.opts.tc_engine == 1)   // the tables are for the tcgen05 engine
            return analytic_cost(1, rows_blk, std::max(1, tokens), bytes_per_tok, P.d, num_sms);
        return cost_us(cost_kind(t), rows_blk, std::max(1, tokens), bytes_per_tok, P.d, num_sms);
    }

    int rows_per_block(const Task& t) const {
        return t.kind == 1 ? tc_rows_per_block(P.opts) : P.thin ? thin_rows(t.rows) : cc_row_tile(t.rows);
    }

    // kv heads one item covers (the thin PAC takes kThinHeads at once)
    int heads_per_item(const Task& t) const { return (t.kind == 0 && P.thin) ? kThinHeads : 1; }

    // C_est of each item of task i split b ways (one per chunk and row
    // block, chunk-major; every kv head's item costs the same). Memoised: the
    // search below scores many partitions that share a task's split count.
    mutable std::vector<std::unordered_map<int, std::vector<double>>> memo;
    const std::vector<double>& task_costs(size_t i, int b) const {
        if (memo.size() != P.tasks.size()) memo.assign(P.tasks.size(), {});
        auto hit = memo[i].find(b);
        if (hit != memo[i].end()) return hit->second;
        const Task& t = P.tasks[i];
        const int rpb = rows_per_block(t);
        const int n_rb = (t.rows + rpb - 1) / rpb;
        Span s = t.node >= 0 ? node_span(T.first_offset[t.node], t.n_tok, tile_tokens(t.kind, P.opts, P.thin))
                              : Span{0, t.n_tok, 0, 1, kTileTokens};
        std::vector<double> c;
        c.reserve((size_t)b * n_rb);
        for (int k = 0; k < b; ++k) {
            int32_t tb = 0, te = t.n_tok;
            if (t.node >= 0) chunk_range(s, b, k, &tb, &te);
            for (int rb = 0; rb < n_rb; ++rb) c.push_back(item_cost(t, std::min(rpb, t.rows - rb * rpb), te - tb));
        }
        return memo[i].emplace(b, std::move(c)).first->second;
    }

    // sum of the item costs of task i split b ways, over the kv heads
    void add_task_total(size_t i, int b, double* total) const {
        const int per = P.hkv / heads_per_item(P.tasks[i]);
        for (double c : task_costs(i, b)) *total += c * per;
    }

    // makespan of split vector b: memoised, since the candidate partitions
    // the search scores often coincide (the factors and the uniform sizes
    // map most tasks to the same split counts)
    struct VecHash {
        size_t operator()(const std::vector<int>& b) const {
            uint64_t h = 1469598103934665603ull;
            for (int x : b) h = (h ^ (uint32_t)x) * 1099511628211ull;
            return (size_t)h;
        }
    };
    mutable std::unordered_map<std::vector<int>, double, VecHash> mk_memo;
    double makespan(const std::vector<int>& b, int m) const {
        auto hit = mk_memo.find(b);
        if (hit != mk_memo.end()) return hit->second;
        const double mk = simulate(b, m);
        mk_memo.emplace(b, mk);
        return mk;
    }
    double simulate(const std::vector<int>& b, int m) const {
        (void)m;
        std::vector<CostRun> v;
        for (size_t i = 0; i < P.tasks.size(); ++i) {
            const Task& t = P.tasks[i];
            const int hpi = heads_per_item(t);
            const int32_t n = (P.hkv + hpi - 1) / hpi;
            const int8_t klass = item_class(t);
            for (double c : task_costs(i, b[i])) v.push_back({c, n, klass});
        }
        return simulate_call(v, num_sms, cc_per_sm);
    }

    // launch class of a task's items (see ItemCost::klass)
    int8_t item_class(const Task& t) const {
        if (t.kind == 1) return (int8_t)((P.opts.tc_engine == 0 && cost_kind(t) == 2) ? 1 : 0);
        if (P.thin) return (int8_t)(t.rows > 4 ? 2 : 3);   // thin PAC row blocks of 8, of 4
        const int rt = cc_row_tile(t.rows);
        return (int8_t)(2 + (rt == 8 ? 0 : rt == 4 ? 1 : rt == 2 ? 2 : 3));
    }

    // CoDec's heuristic solver: binary search for cost_l, bound b_k, then a
    // search over the bounded b_k vectors scored by the list schedule.
    void partition(int m) {
        auto& tasks = P.tasks;
        const size_t nt = tasks.size();
        std::vector<double> c_full(nt);
        for (size_t i = 0; i < nt; ++i) c_full[i] = item_cost(tasks[i], rows_per_block(tasks[i]), tasks[i].n_tok);
        auto b_of = [&](size_t i, double Tc, int cap) {
            if (Tc <= 0) return cap;
            int b = (int)std::ceil(c_full[i] / Tc - 1e-9);
            return std::max(1, std::min(b, cap));
        };
        auto avg_at = [&](double Tc) {
            double total = 0;
            for (size_t i = 0; i < nt; ++i) add_task_total(i, b_of(i, Tc, tasks[i].max_splits), &total);
            return total / m;
        };
        double hi = 0, lo = 1e30;
        for (size_t i = 0; i < nt; ++i) {
            hi = std::max(hi, c_full[i]);
            lo = std::min(lo, item_cost(tasks[i], rows_per_block(tasks[i]), std::min(tasks[i].n_tok, kTileTokens)));
        }
        double cost_l;
        const double avg_hi = avg_at(hi);
        if (avg_hi >= hi) {
            cost_l = avg_hi;  // coarsest split already averages above the largest task
        } else {
            lo = std::min(lo, hi);
            for (int it = 0; it < 60 && hi - lo > 1e-4 * hi; ++it) {
                const double mid = 0.5 * (lo + hi);
                if (avg_at(mid) <= mid) hi = mid; else lo = mid;
            }
            cost_l = hi;
        }
        P.cost_l_us = cost_l;
        std::vector<int> ub(nt);
        for (size_t i = 0; i < nt; ++i) ub[i] = b_of(i, cost_l, tasks[i].max_splits);

        std::vector<int> best(nt, 1);
        double best_mk = 1e300;
        const double factors[] = {0.6, 0.7, 0.8, 0.9, 1.0, 1.15, 1.3, 1.5, 2.0, 3.0};
        auto consider = [&](const std::vector<int>& b) {
            const double mk = makespan(b, m);
            if (mk < best_mk * (1 - 1e-9)) { best_mk = mk; best = b; }
        };
        for (double f : factors) {
            std::vector<int> b(nt);
            for (size_t i = 0; i < nt; ++i) b[i] = b_of(i, cost_l * f, ub[i]);
            consider(b);
        }
        // the plan is never worse (under C_est) than no split or a uniform split
        consider(std::vector<int>(nt, 1));
        // (64, 128, 192, 256, 384, ... 6144, 8192 tokens: powers of two and
        // their halfway points, all multiples of the 64-token tile)
        for (int pow2 = kTileTokens; pow2 <= 8192; pow2 *= 2) {
            for (int chunk : {pow2, pow2 * 3 / 2}) {
                if (chunk > 8192 || chunk % kTileTokens) continue;
                std::vector<int> b(nt);
                for (size_t i = 0; i < nt; ++i)
                    b[i] = tasks[i].node < 0 ? 1
                                             : std::max(1, std::min(tasks[i].max_splits, (tasks[i].n_tok + chunk - 1) / chunk));
                consider(b);
            }
        }
        // greedy +-1 refinement of single tasks, largest per-item cost first
        for (int iter = 0; iter < 24; ++iter) {
            std::vector<size_t> order(nt);
            std::iota(order.begin(), order.end(), 0);
            std::sort(order.begin(), order.end(), [&](size_t a, size_t b2) {
                double ca = c_full[a] / best[a], cb = c_full[b2] / best[b2];
                return ca != cb ? ca > cb : a < b2;
            });
            bool improved = false;
            for (size_t k = 0; k < std::min<size_t>(order.size(), 4) && !improved; ++k) {
                const size_t i = order[k];
                for (int delta : {+1, -1}) {
                    const int nb = best[i] + delta;
                    if (nb < 1 || nb > tasks[i].max_splits) continue;
                    std::vector<int> b = best;
                    b[i] = nb;
                    const double mk = makespan(b, m);
                    if (mk < best_mk * (1 - 1e-6)) { best_mk = mk; best = b; improved = true; break; }
                }
            }
            if (!improved) break;
        }
        for (size_t i = 0; i < nt; ++i) tasks[i].b_k = best[i];
        P.makespan_us = best_mk;
    }
};

static bool build_packed_group(const Tree& T, int32_t root, const std::vector<int32_t>& desc,
                               PackedGroup* g) {
    // Try chunk orders: ascending node id (allocation order), then preorder.
    std::vector<std::vector<int32_t>> orders;
    std::vector<int32_t> by_id = desc;
    std::sort(by_id.begin(), by_id.end());
    orders.push_back(by_id);
    orders.push_back(desc);  // desc is in preorder
    const int32_t ps = T.page_size;
    for (const auto& ord : orders) {
        std::vector<int32_t> plist, tn, tt;
        int32_t pos_begin = -1, cur_page = -1, cur_row = -1;
        bool ok = true;
        for (int32_t n : ord) {
            for (int32_t t = 0; t < T.len[n] && ok; ++t) {
                const int64_t pos = (int64_t)T.first_offset[n] + t;
                const int32_t page = T.page_ids[T.page_ptr[n] + pos / ps];
                const int32_t row = (int32_t)(pos % ps);
                if (cur_page < 0) {
                    plist.push_back(page);
                    pos_begin = row;
                } else if (page == cur_page && row == cur_row + 1) {
                    // continues in the same page
                } else if (cur_row == ps - 1 && row == 0) {
                    plist.push_back(page);
                } else {
                    ok = false;
                }
                cur_page = page;
                cur_row = row;
                tn.push_back(n);
                tt.push_back(t);
            }
            if (!ok) break;
        }
        if (!ok || tn.empty()) continue;
        g->root = root;
        g->nodes = ord;
        g->tok_node = std::move(tn);
        g->tok_t = std::move(tt);
        g->page_list = std::move(plist);
        g->pos_begin = pos_begin;
        return true;
    }
    return false;
}

// Plan creation; with `prev` the KV-axis splits are taken from it instead of
// being searched (pst_plan_update). With `score_only` the build stops once
// the predicted makespan is known: a DEFT-Flatten run then keeps its token
// count, nodes and queries, not its per-token records or masks, and no
// chunks, items or metadata are made (the plan is good for its makespan only).
static int plan_build(const pst_tree* tree, int32_t n_queries, const int32_t* query_node, int32_t n_q_heads,
                      int32_t n_kv_heads, int32_t d, pst_dtype dtype, const pst_plan_opts* opts,
                      const pst_plan* prev, const int32_t* prev_node, pst_plan** out, bool score_only = false) {
    const auto t_start = std::chrono::steady_clock::now();
    if (!out) return fail(PST_EINVAL, "plan_create: out is null");
    *out = nullptr;
    if (!tree) return fail(PST_EINVAL, "plan_create: tree is null");
    if (n_queries < 1 || !query_node) return fail(PST_EINVAL, "plan_create: need >= 1 query");
    if (n_q_heads < 1 || n_kv_heads < 1 || n_q_heads % n_kv_heads)
        return fail(PST_EUNSUPPORTED, "plan_create: n_q_heads must be a positive multiple of n_kv_heads");
    if (n_q_heads > 32767 || n_kv_heads > 32767) return fail(PST_EUNSUPPORTED, "plan_create: too many heads");
    if (d != 64 && d != 128) return fail(PST_EUNSUPPORTED, "plan_create: d must be 64 or 128");
    if (dtype != PST_BF16 && dtype != PST_F32) return fail(PST_EUNSUPPORTED, "plan_create: dtype");
    const Tree& T = tree->t;
    pst_plan_opts o;
    pst_plan_opts_default(&o);
    if (opts) o = *opts;
    if (o.tc_min_rows <= 0) o.tc_min_rows = 16;
    if (o.slots_per_sm <= 0) o.slots_per_sm = 1;
    if (o.tc_block_rows != 128) o.tc_block_rows = 256;
    if (o.p_bf16_min_tokens == 0) o.p_bf16_min_tokens = kPBf16MinTokens;
    if (o.split_policy == PST_SPLIT_UNIFORM && (o.fixed_chunk <= 0 || o.fixed_chunk % kTileTokens))
        return fail(PST_EINVAL, "plan_create: fixed_chunk must be a positive multiple of 64");
    if (o.split_policy == PST_SPLIT_FLATTEN && o.fixed_chunk <= 0) o.fixed_chunk = kMaskTokens;
    if (o.split_policy < PST_SPLIT_COST_MODEL || o.split_policy > PST_SPLIT_FLATTEN)
        return fail(PST_EINVAL, "plan_create: unknown split policy");

    pst_plan* P = new (std::nothrow) pst_plan();
    if (!P) return fail(PST_ENOMEM, "plan_create: out of memory");
    std::unique_ptr<pst_plan> guard(P);
    P->n_queries = n_queries;
    P->hq = n_q_heads;
    P->hkv = n_kv_heads;
    P->group = n_q_heads / n_kv_heads;
    P->d = d;
    P->dtype = dtype;
    P->page_size = T.page_size;
    P->num_pages = T.num_pages;
    P->n_nodes = T.n_nodes;
    P->opts = o;
    P->thin = dtype == PST_BF16 && d == 128 && n_kv_heads % kThinHeads == 0 && o.thin_engine == 0;
    const int32_t N = T.n_nodes, G = P->group;

    // ---- QMapKV: per query, its path from the top of its tree (DEFT Alg. 1 step 1)
    P->qpath_ptr.assign(n_queries + 1, 0);
    for (int32_t q = 0; q < n_queries; ++q) {
        const int32_t v = query_node[q];
        if (v < 0 || v >= N) return fail(PST_EINVAL, "plan_create: query " + std::to_string(q) + " node out of range");
        P->qpath_ptr[q + 1] = P->qpath_ptr[q] + T.depth[v] + 1;
    }
    P->qpath_node.resize(P->qpath_ptr[n_queries]);
    for (int32_t q = 0; q < n_queries; ++q) {
        int32_t k = P->qpath_ptr[q + 1];
        int64_t seen = 0;
        for (int32_t n = query_node[q]; n >= 0; n = T.parent[n]) {
            P->qpath_node[--k] = n;
            seen += T.len[n];
        }
        if (seen == 0) return fail(PST_EINVAL, "plan_create: query " + std::to_string(q) + " sees no token");
    }
    // ---- KVMapQ: per node, ascending queries sharing it (DEFT Alg. 1 step 2)
    P->nodeq_ptr.assign(N + 1, 0);
    for (int32_t n : P->qpath_node) P->nodeq_ptr[n + 1]++;
    for (int32_t n = 0; n < N; ++n) P->nodeq_ptr[n + 1] += P->nodeq_ptr[n];
    P->nodeq.resize(P->nodeq_ptr[N]);
    {
        std::vector<int32_t> fill(P->nodeq_ptr.begin(), P->nodeq_ptr.end() - 1);
        for (int32_t q = 0; q < n_queries; ++q)
            for (int32_t k = P->qpath_ptr[q]; k < P->qpath_ptr[q + 1]; ++k)
                P->nodeq[fill[P->qpath_node[k]]++] = q;
    }
    auto nq_of = [&](int32_t n) { return P->nodeq_ptr[n + 1] - P->nodeq_ptr[n]; };

    // A packed chunk's queries (the union of the query lists of `nodes`) and
    // the bit causal mask of each: bit j set iff chunk token j's node is on
    // the query's path (DEFT, section 3.3 and A.9).
    auto set_queries_and_masks = [&](PackedGroup& g, const std::vector<int32_t>& nodes, bool with_masks) {
        std::vector<int32_t> qs;
        for (int32_t n : nodes)
            qs.insert(qs.end(), P->nodeq.begin() + P->nodeq_ptr[n], P->nodeq.begin() + P->nodeq_ptr[n + 1]);
        std::sort(qs.begin(), qs.end());
        qs.erase(std::unique(qs.begin(), qs.end()), qs.end());
        g.queries = qs;
        g.mask.clear();
        if (!with_masks) return;
        g.mask.assign(qs.size(), 0);
        for (size_t qi = 0; qi < qs.size(); ++qi) {
            const int32_t q = qs[qi];
            uint64_t m = 0;
            for (size_t j = 0; j < g.tok_node.size(); ++j) {
                bool on = false;
                for (int32_t k = P->qpath_ptr[q]; k < P->qpath_ptr[q + 1]; ++k)
                    if (P->qpath_node[k] == g.tok_node[j]) { on = true; break; }
                if (on) m |= (uint64_t)1 << j;
            }
            g.mask[qi] = m;
        }
    };

    // ---- packing: a page-contiguous set of descendants of <= 64 tokens
    std::vector<int32_t> packed_in(N, -1);
    std::vector<int32_t> run_tokens;   // tokens of each DEFT-Flatten run (groups made below)
    if (o.split_policy == PST_SPLIT_FLATTEN) {
        // DEFT-Flatten: walk the nodes some query sees in depth-first order
        // and cut their tokens into runs of at most fixed_chunk (S_t); a run
        // that mixes nodes needs a mask bit per token, so it holds at most 64;
        // a run also ends where the next token is not the next page row (the
        // kernels read a chunk as consecutive rows of its page list). A run
        // inside one node needs no mask: all of the node's queries see all of
        // its tokens.
        const int32_t ps = T.page_size;
        PackedGroup cur;
        int32_t cur_page = -1, cur_row = -1;
        int32_t held_tok = 0;   // tokens in the run so far
        auto flush = [&]() {
            if (held_tok == 0) return;
            cur.root = -1;
            if (!score_only) {
                cur.nodes.clear();   // the run's nodes, in walk order (each node's tokens are consecutive)
                for (int32_t n : cur.tok_node)
                    if (cur.nodes.empty() || cur.nodes.back() != n) cur.nodes.push_back(n);
            }
            // one node: every query sees every token, no mask (and the run may
            // be longer than the 64 bits of one)
            set_queries_and_masks(cur, cur.nodes, !score_only && cur.nodes.size() > 1);
            const int32_t gid = (int32_t)P->groups.size();
            for (int32_t n : cur.nodes) packed_in[n] = gid;   // every flattened node is in some run
            run_tokens.push_back(held_tok);
            P->groups.push_back(std::move(cur));
            cur = PackedGroup();
            held_tok = 0;
        };
        // tokens [t0, t0 + k) of node n join the run, a page row-range at a time
        auto append = [&](int32_t n, int32_t t0, int32_t k) {
            if (score_only) {   // the count, the nodes and where the run ends
                if (cur.nodes.empty() || cur.nodes.back() != n) cur.nodes.push_back(n);
                const int64_t last = (int64_t)T.first_offset[n] + t0 + k - 1;
                cur_page = T.page_ids[T.page_ptr[n] + last / ps];
                cur_row = (int32_t)(last % ps);
                held_tok += k;
                return;
            }
            held_tok += k;
            for (int32_t t = t0; t < t0 + k;) {
                const int64_t pos = (int64_t)T.first_offset[n] + t;
                const int32_t page = T.page_ids[T.page_ptr[n] + pos / ps];
                const int32_t row = (int32_t)(pos % ps);
                const int32_t m = std::min(t0 + k - t, ps - row);
                if (cur.tok_node.empty()) {
                    cur.page_list.assign(1, page);
                    cur.pos_begin = row;
                } else if (page != cur_page) {
                    cur.page_list.push_back(page);
                }
                cur.tok_node.insert(cur.tok_node.end(), m, n);
                for (int32_t j = 0; j < m; ++j) cur.tok_t.push_back(t + j);
                cur_page = page;
                cur_row = row + m - 1;
                t += m;
            }
        };
        for (int i = 0; i < N; ++i) {
            const int32_t n = T.preorder[i];
            if (T.len[n] == 0 || nq_of(n) == 0) continue;
            // A node's tokens follow one another on its pages (the next row, or
            // row 0 after the last row), so within the node a run ends only at
            // its length limit; the first token may also end it for want of
            // page continuity with the run so far.
            for (int32_t t = 0; t < T.len[n];) {
                const int64_t pos = (int64_t)T.first_offset[n] + t;
                const int32_t page = T.page_ids[T.page_ptr[n] + pos / ps];
                const int32_t row = (int32_t)(pos % ps);
                int32_t held = held_tok;
                const bool next_row = held > 0 &&
                                      ((page == cur_page && row == cur_row + 1) || (cur_row == ps - 1 && row == 0));
                // joining this token to the run would make it mix nodes (the
                // walk visits each node's tokens in one stretch)
                const bool mixes = held > 0 && (score_only ? cur.nodes.front() : cur.tok_node.front()) != n;
                int32_t limit = mixes ? std::min(o.fixed_chunk, kMaskTokens) : o.fixed_chunk;
                if (held > 0 && (!next_row || held >= limit)) {
                    flush();
                    held = 0;
                    limit = o.fixed_chunk;
                }
                const int32_t k = std::min(T.len[n] - t, limit - held);
                append(n, t, k);
                t += k;
            }
        }
        flush();
    } else if (o.pack_masks) {
        // subtree token totals (excluding the node itself) via reverse preorder
        std::vector<int64_t> sub_tok(N, 0), sub_cnt(N, 0);
        for (int i = N - 1; i >= 0; --i) {
            const int32_t n = T.preorder[i];
            for (int32_t c : T.children[n]) {
                sub_tok[n] += sub_tok[c] + T.len[c];
                sub_cnt[n] += sub_cnt[c] + 1;
            }
        }
        for (int i = 0; i < N; ++i) {
            const int32_t p = T.preorder[i];
            if (packed_in[p] >= 0) continue;
            if (sub_cnt[p] < 2 || sub_tok[p] < 2 || sub_tok[p] > kMaskTokens) continue;
            // descendants in preorder
            std::vector<int32_t> desc, st(T.children[p].rbegin(), T.children[p].rend());
            while (!st.empty()) {
                int32_t n = st.back();
                st.pop_back();
                desc.push_back(n);
                for (auto it = T.children[n].rbegin(); it != T.children[n].rend(); ++it) st.push_back(*it);
            }
            PackedGroup g;
            if (!build_packed_group(T, p, desc, &g)) continue;
            set_queries_and_masks(g, desc, true);
            if (g.queries.empty()) continue;
            const int32_t gid = (int32_t)P->groups.size();
            for (int32_t n : desc) packed_in[n] = gid;
            P->groups.push_back(std::move(g));
        }
    }

    // ---- tasks T[i] = (n_q[i], n[i])
    const bool tc_ok = dtype == PST_BF16;
    for (int i = 0; i < N; ++i) {
        const int32_t n = T.preorder[i];
        if (packed_in[n] >= 0 || T.len[n] == 0 || nq_of(n) == 0) continue;
        Task t;
        t.node = n;
        t.group = -1;
        t.n_q = nq_of(n);
        t.rows = t.n_q * G;
        t.n_tok = T.len[n];
        t.kind = (tc_ok && t.rows >= o.tc_min_rows) ? 1 : 0;
        t.max_splits = node_span(T.first_offset[n], T.len[n], tile_tokens(t.kind, o, P->thin)).n_blocks;
        P->tasks.push_back(t);
    }
    for (size_t gi = 0; gi < P->groups.size(); ++gi) {
        const auto& g = P->groups[gi];
        Task t;
        t.node = -1;
        t.group = (int32_t)gi;
        t.n_q = (int32_t)g.queries.size();
        t.rows = t.n_q * G;
        t.n_tok = gi < run_tokens.size() ? run_tokens[gi] : (int32_t)g.tok_node.size();
        t.kind = (tc_ok && t.rows >= o.tc_min_rows) ? 1 : 0;
        t.max_splits = 1;
        P->tasks.push_back(t);
    }

    // ---- partition (b_k)
    Planner pl(T, *P);
    if (o.num_sms > 0) pl.num_sms = o.num_sms;
    else {
        int sms = 0;
        if (device_sm_count(&sms) != 0 || sms <= 0) return fail(PST_ECUDA, "plan_create: cannot query the SM count (set opts.num_sms)");
        pl.num_sms = sms;
    }
    pl.bytes_per_tok = 2.0 * d * (dtype == PST_BF16 ? 2 : 4);
    if (P->thin) {
        pl.cc_per_sm[0] = pl.cc_per_sm[1] = 1;
    } else {
        for (int k = 0; k < 4; ++k) {
            const int n = pst::cc_blocks_per_sm(dtype, d, 8 >> k);
            if (n > 0) pl.cc_per_sm[k] = n;
        }
    }
    const int m = pl.num_sms * o.slots_per_sm;
    P->num_slots = m;
    if (prev) {
        // CoDec reuses a plan across decode steps: a node keeps its previous
        // split b_k (bounded by its tiles now); a node that is new (or a
        // packing that changed) gets the split its cost bound under the
        // previous cost_l gives, ceil(C_est / cost_l). prev_node maps a node
        // to its id in prev's tree (-1: new); null means the same ids.
        std::vector<int32_t> bk_of_old(prev->n_nodes, 0);
        for (const auto& t : prev->tasks)
            if (t.node >= 0 && t.node < prev->n_nodes) bk_of_old[t.node] = t.b_k;
        P->cost_l_us = prev->cost_l_us;
        for (auto& t : P->tasks) {
            int32_t b = 1;
            if (t.node >= 0) {
                const int32_t old_id = prev_node ? prev_node[t.node] : t.node;
                b = (old_id >= 0 && old_id < prev->n_nodes) ? bk_of_old[old_id] : 0;
            }
            if (b <= 0) {
                const double c = pl.item_cost(t, pl.rows_per_block(t), t.n_tok);
                b = prev->cost_l_us > 0 ? (int32_t)std::ceil(c / prev->cost_l_us - 1e-9) : 1;
            }
            t.b_k = std::max(1, std::min(b, t.max_splits));
        }
    } else if (o.split_policy == PST_SPLIT_NONE) {
        for (auto& t : P->tasks) t.b_k = 1;
    } else if (o.split_policy == PST_SPLIT_UNIFORM) {
        for (auto& t : P->tasks)
            t.b_k = t.node < 0 ? 1 : std::max(1, std::min(t.max_splits, (t.n_tok + o.fixed_chunk - 1) / o.fixed_chunk));
    } else {
        pl.partition(m);
    }
    {
        std::vector<int> b(P->tasks.size());
        for (size_t i = 0; i < b.size(); ++i) b[i] = P->tasks[i].b_k;
        P->makespan_us = pl.makespan(b, m);
    }
    if (score_only) {
        *out = guard.release();
        return PST_OK;
    }

    // ---- chunks, pages, chunk queries, masks, partial rows
    P->pages = T.page_ids;
    int64_t part_rows = 0;
    for (size_t ti = 0; ti < P->tasks.size(); ++ti) {
        const Task& t = P->tasks[ti];
        if (t.node >= 0) {
            Span s = node_span(T.first_offset[t.node], t.n_tok, tile_tokens(t.kind, o, P->thin));
            for (int k = 0; k < t.b_k; ++k) {
                int32_t tb, te;
                chunk_range(s, t.b_k, k, &tb, &te);
                if (te <= tb) continue;
                HostChunk c;
                c.task = (int32_t)ti;
                c.node = t.node;
                c.tok_begin = tb;
                c.tok_end = te;
                c.kind = t.kind;
                c.dev.page_base = (int32_t)T.page_ptr[t.node];
                c.dev.pos_begin = T.first_offset[t.node] + tb;
                c.dev.n_tok = te - tb;
                c.dev.q_base = (int32_t)P->chunk_q.size();
                c.dev.n_q = t.n_q;
                c.dev.mask_base = -1;
                c.dev.r_tile = pl.rows_per_block(t);
                P->chunk_q.insert(P->chunk_q.end(), P->nodeq.begin() + P->nodeq_ptr[t.node],
                                  P->nodeq.begin() + P->nodeq_ptr[t.node + 1]);
                P->chunks.push_back(c);
            }
        } else {
            const PackedGroup& g = P->groups[t.group];
            HostChunk c;
            c.task = (int32_t)ti;
            c.node = -1;
            c.tok_begin = 0;
            c.tok_end = t.n_tok;
            c.kind = t.kind;
            c.dev.page_base = (int32_t)P->pages.size();
            P->pages.insert(P->pages.end(), g.page_list.begin(), g.page_list.end());
            c.dev.pos_begin = g.pos_begin;
            c.dev.n_tok = t.n_tok;
            c.dev.q_base = (int32_t)P->chunk_q.size();
            c.dev.n_q = t.n_q;
            c.dev.mask_base = g.mask.empty() ? -1 : (int32_t)P->masks.size();
            c.dev.r_tile = pl.rows_per_block(t);
            P->chunk_q.insert(P->chunk_q.end(), g.queries.begin(), g.queries.end());
            P->masks.insert(P->masks.end(), g.mask.begin(), g.mask.end());
            P->chunks.push_back(c);
        }
    }
    for (auto& c : P->chunks) {
        c.dev.part_base = (int32_t)part_rows;
        part_rows += (int64_t)c.dev.n_q * n_q_heads;
        // tokens the kernel loads (whole 16-row boxes)
        const int32_t b0 = c.dev.pos_begin / kBoxRows, b1 = (c.dev.pos_begin + c.dev.n_tok + kBoxRows - 1) / kBoxRows;
        P->kv_tokens_read += (int64_t)(b1 - b0) * kBoxRows;
    }
    if (part_rows > INT32_MAX) return fail(PST_EUNSUPPORTED, "plan_create: too many partial rows");
    P->n_part_rows = part_rows;
    for (int32_t n = 0; n < N; ++n) P->unique_tokens += T.len[n];

    // ---- merge lists: per query, the partial rows POR combines
    P->merge_ptr.assign(n_queries + 1, 0);
    for (const auto& c : P->chunks)
        for (int32_t k = 0; k < c.dev.n_q; ++k) P->merge_ptr[P->chunk_q[c.dev.q_base + k] + 1]++;
    for (int32_t q = 0; q < n_queries; ++q) P->merge_ptr[q + 1] += P->merge_ptr[q];
    P->merge_row.resize(P->merge_ptr[n_queries]);
    {
        std::vector<int32_t> fill(P->merge_ptr.begin(), P->merge_ptr.end() - 1);
        for (const auto& c : P->chunks)
            for (int32_t k = 0; k < c.dev.n_q; ++k)
                P->merge_row[fill[P->chunk_q[c.dev.q_base + k]]++] = c.dev.part_base + k * n_q_heads;
    }

    // ---- items in largest-first order (the hardware block dispatcher then
    // realises a list schedule of them), tensor-core items first
    std::vector<ItemCost> tc, cc;
    for (size_t ci = 0; ci < P->chunks.size(); ++ci) {
        const auto& c = P->chunks[ci];
        const Task& t = P->tasks[c.task];
        const int rpb = pl.rows_per_block(t);
        const int n_rb = (t.rows + rpb - 1) / rpb;
        for (int rb = 0; rb < n_rb; ++rb) {
            const int rows_blk = std::min(rpb, t.rows - rb * rpb);
            const double cst = pl.item_cost(t, rows_blk, c.dev.n_tok);
            for (int h = 0; h < n_kv_heads; h += pl.heads_per_item(t))
                (t.kind == 1 ? tc : cc).push_back({cst, (int32_t)ci, (int16_t)h, (int16_t)rb, pl.item_class(t)});
        }
    }
    list_schedule(tc, m);
    list_schedule(cc, m);
    // tensor-core launch groups (see pst_plan::tc_group_cnt): precision, then
    // row-block mode. The rounding errors of a node's chunks average out in
    // POR like those inside one chunk, so the node's length decides the
    // precision.
    const int32_t p_single = o.p_bf16_min_tokens < 0 ? INT32_MAX : o.p_bf16_min_tokens;
    auto tc_group = [&](const ItemCost& it) {
        const HostChunk& hc = P->chunks[it.chunk];
        const bool exact = o.tc_engine == 0 && P->tasks[hc.task].n_tok < p_single;
        const int rows_total = hc.dev.n_q * G;
        const bool split = o.tc_engine == 0 && std::min(hc.dev.r_tile, rows_total - it.rb * hc.dev.r_tile) > 128;
        return (exact ? 2 : 0) + (split ? 0 : 1);
    };
    for (int g = 0; g < 4; ++g) {
        const size_t before = P->items.size();
        for (const auto& it : tc)
            if (tc_group(it) == g) P->items.push_back({it.chunk, it.head, it.rb});
        P->tc_group_cnt[g] = (int64_t)(P->items.size() - before);
    }
    P->n_tc_items = (int64_t)tc.size();
    P->n_cc_items = (int64_t)cc.size();
    // thin chunks: one launch of the thin PAC, or one CUDA-core launch per row
    // tile (8, 4, 2, 1); each in largest-first order
    for (int k = 0; k < 4; ++k) {
        P->cc_class_off[k] = (int64_t)P->items.size();
        for (const auto& it : cc)
            if (it.klass - 2 == k) P->items.push_back({it.chunk, it.head, it.rb});
        P->cc_class_cnt[k] = (int64_t)P->items.size() - P->cc_class_off[k];
    }

    // ---- workspace layout and the metadata image
    WsLayout& W = P->ws;
    int64_t off = 0;
    W.status = off; off = align256(off + 64);
    W.items = off; off = align256(off + (int64_t)P->items.size() * sizeof(DevItem));
    W.chunks = off; off = align256(off + (int64_t)P->chunks.size() * sizeof(DevChunk));
    W.pages = off; off = align256(off + (int64_t)P->pages.size() * 4);
    W.chunk_q = off; off = align256(off + (int64_t)P->chunk_q.size() * 4);
    W.masks = off; off = align256(off + (int64_t)P->masks.size() * 8);
    W.merge_ptr = off; off = align256(off + (int64_t)P->merge_ptr.size() * 4);
    W.merge_row = off; off = align256(off + (int64_t)P->merge_row.size() * 4);
    P->tree_pages = T.unique_pages;
    W.tree_pages = off; off = align256(off + (int64_t)P->tree_pages.size() * 4);
    W.meta_end = off;
    W.part_o = off; off = align256(off + part_rows * d * 4);
    W.part_lse = off; off = align256(off + part_rows * 4);
    W.total = off;
    P->meta_blob.assign(W.meta_end, 0);
    auto put = [&](int64_t at, const void* src, size_t n) { if (n) std::memcpy(P->meta_blob.data() + at, src, n); };
    put(W.items, P->items.data(), P->items.size() * sizeof(DevItem));
    {
        std::vector<DevChunk> dc(P->chunks.size());
        for (size_t i = 0; i < dc.size(); ++i) dc[i] = P->chunks[i].dev;
        put(W.chunks, dc.data(), dc.size() * sizeof(DevChunk));
    }
    put(W.pages, P->pages.data(), P->pages.size() * 4);
    put(W.chunk_q, P->chunk_q.data(), P->chunk_q.size() * 4);
    put(W.masks, P->masks.data(), P->masks.size() * 8);
    put(W.merge_ptr, P->merge_ptr.data(), P->merge_ptr.size() * 4);
    put(W.merge_row, P->merge_row.data(), P->merge_row.size() * 4);
    put(W.tree_pages, P->tree_pages.data(), P->tree_pages.size() * 4);

    P->plan_us = std::chrono::duration<double, std::micro>(std::chrono::steady_clock::now() - t_start).count();
    *out = guard.release();
    return PST_OK;
}

// CoDec keeps the candidate partition its cost model scores best; the
// cost-model policy also scores DEFT-Flatten chunkings (DEFT A.9) of these
// sizes and takes one only when its predicted makespan is lower by the margin:
// measured on GB300, the model ranks node partitions and flattened plans in
// the right order, but its error is larger on flattened plans.
static constexpr int32_t kFlattenCandidates[] = {1024, 2048};
static constexpr double kFlattenMargin = 0.97;

extern "C" int pst_plan_create(const pst_tree* tree, int32_t n_queries, const int32_t* query_node,
                               int32_t n_q_heads, int32_t n_kv_heads, int32_t d, pst_dtype dtype,
                               const pst_plan_opts* opts, pst_plan** out) {
    const auto t0 = std::chrono::steady_clock::now();
    int rc = plan_build(tree, n_queries, query_node, n_q_heads, n_kv_heads, d, dtype, opts, nullptr, nullptr, out);
    if (rc != PST_OK) return rc;
    if ((*out)->opts.split_policy != PST_SPLIT_COST_MODEL || (*out)->opts.flatten_candidates < 0) return rc;
    // score each candidate without building it; build the winner, if any
    const double ref = (*out)->makespan_us;   // the node partition's
    double best_mk = ref;
    int32_t best_st = 0;
    for (int32_t st : kFlattenCandidates) {
        pst_plan_opts fo = (*out)->opts;
        fo.split_policy = PST_SPLIT_FLATTEN;
        fo.fixed_chunk = st;
        pst_plan* alt = nullptr;
        if (plan_build(tree, n_queries, query_node, n_q_heads, n_kv_heads, d, dtype, &fo, nullptr, nullptr, &alt,
                       true) != PST_OK)
            continue;
        if (alt->makespan_us < kFlattenMargin * ref && alt->makespan_us < best_mk) {
            best_mk = alt->makespan_us;
            best_st = st;
        }
        pst_plan_destroy(alt);
    }
    if (best_st > 0) {
        pst_plan_opts fo = (*out)->opts;
        fo.split_policy = PST_SPLIT_FLATTEN;
        fo.fixed_chunk = best_st;
        pst_plan* alt = nullptr;
        if (plan_build(tree, n_queries, query_node, n_q_heads, n_kv_heads, d, dtype, &fo, nullptr, nullptr, &alt) ==
            PST_OK) {
            pst_plan_destroy(*out);
            *out = alt;
        }
    }
    (*out)->plan_us = std::chrono::duration<double, std::micro>(std::chrono::steady_clock::now() - t0).count();
    return PST_OK;
}

extern "C" int pst_plan_update(const pst_plan* prev, const pst_tree* tree, pst_plan** out) {
    if (!out) return fail(PST_EINVAL, "plan_update: out is null");
    *out = nullptr;
    if (!prev || !tree) return fail(PST_EINVAL, "plan_update: null plan or tree");
    const Tree& T = tree->t;
    if (T.n_nodes != prev->n_nodes) return fail(PST_EINVAL, "plan_update: the tree has a different node count");
    // the queries sit where they sat: the last node of each query's path
    std::vector<int32_t> qn(prev->n_queries);
    for (int32_t q = 0; q < prev->n_queries; ++q) qn[q] = prev->qpath_node[prev->qpath_ptr[q + 1] - 1];
    // the node structure must be the same: every query's path is unchanged
    for (int32_t q = 0; q < prev->n_queries; ++q) {
        int32_t v = qn[q];
        for (int32_t k = prev->qpath_ptr[q + 1] - 1; k >= prev->qpath_ptr[q]; --k) {
            if (v < 0 || prev->qpath_node[k] != v) return fail(PST_EINVAL, "plan_update: the tree's parents changed");
            v = T.parent[v];
        }
        if (v != -1) return fail(PST_EINVAL, "plan_update: the tree's parents changed");
    }
    return plan_build(tree, prev->n_queries, qn.data(), prev->hq, prev->hkv, prev->d, prev->dtype, &prev->opts, prev,
                      nullptr, out);
}

extern "C" int pst_plan_update_tree(const pst_plan* prev, const pst_tree* tree, int32_t n_queries,
                                    const int32_t* query_node, const int32_t* prev_node, pst_plan** out) {
    if (!out) return fail(PST_EINVAL, "plan_update_tree: out is null");
    *out = nullptr;
    if (!prev || !tree || !prev_node) return fail(PST_EINVAL, "plan_update_tree: null plan, tree or node map");
    const Tree& T = tree->t;
    for (int32_t n = 0; n < T.n_nodes; ++n)
        if (prev_node[n] < -1 || prev_node[n] >= prev->n_nodes)
            return fail(PST_ERANGE, "plan_update_tree: prev_node[" + std::to_string(n) + "] out of range");
    return plan_build(tree, n_queries, query_node, prev->hq, prev->hkv, prev->d, prev->dtype, &prev->opts, prev,
                      prev_node, out);
}

namespace pst {
void release_plan_streams(pst_plan* p);  // attn.cu
}
extern "C" void pst_plan_destroy(pst_plan* p) {
    if (!p) return;
    pst::release_plan_streams(p);
    delete p;
}

extern "C" int64_t pst_plan_workspace_bytes(const pst_plan* p) { return p ? p->ws.total : -1; }

extern "C" int pst_plan_stats_get(const pst_plan* p, pst_plan_stats* s) {
    if (!p || !s) return fail(PST_EINVAL, "plan_stats: null argument");
    s->plan_us = p->plan_us;
    s->predicted_makespan_us = p->makespan_us;
    s->cost_lower_bound_us = p->cost_l_us;
    s->n_chunks = (int64_t)p->chunks.size();
    s->n_items = (int64_t)p->items.size();
    s->n_tc_items = p->n_tc_items;
    s->n_cc_items = p->n_cc_items;
    s->n_partial_rows = p->n_part_rows;
    s->unique_kv_tokens = p->unique_tokens;
    s->kv_tokens_read = p->kv_tokens_read;
    s->workspace_bytes = p->ws.total;
    s->num_slots = p->num_slots;
    s->n_launches = 1;
    for (int g = 0; g < 4; ++g) s->n_launches += p->tc_group_cnt[g] > 0;
    for (int k = 0; k < 4; ++k) s->n_launches += p->cc_class_cnt[k] > 0;
    s->split_policy = p->opts.split_policy;
    s->fixed_chunk = p->opts.fixed_chunk;
    return PST_OK;
}

extern "C" int pst_plan_export_sizes(const pst_plan* p, pst_export_sizes* s) {
    if (!p || !s) return fail(PST_EINVAL, "plan_export_sizes: null argument");
    s->n_queries = p->n_queries;
    s->n_nodes = p->n_nodes;
    s->n_chunks = (int64_t)p->chunks.size();
    s->n_qpath = (int64_t)p->qpath_node.size();
    s->n_nodeq = (int64_t)p->nodeq.size();
    s->n_chunk_q = (int64_t)p->chunk_q.size();
    int64_t nt = 0;
    for (const auto& c : p->chunks) nt += c.dev.n_tok;
    s->n_chunk_tok = nt;
    s->n_merge = (int64_t)p->merge_row.size();
    return PST_OK;
}

extern "C" int pst_plan_export(const pst_plan* p, pst_export* e) {
    if (!p || !e) return fail(PST_EINVAL, "plan_export: null argument");
    auto cp = [](int32_t* dst, const std::vector<int32_t>& v) { if (dst && !v.empty()) std::memcpy(dst, v.data(), v.size() * 4); };
    cp(e->qpath_ptr, p->qpath_ptr);
    cp(e->qpath_node, p->qpath_node);
    cp(e->nodeq_ptr, p->nodeq_ptr);
    cp(e->nodeq, p->nodeq);
    cp(e->chunk_q, p->chunk_q);
    cp(e->merge_ptr, p->merge_ptr);
    cp(e->merge_row, p->merge_row);
    int32_t qacc = 0, tacc = 0;
    int64_t tk = 0, qk = 0;
    const size_t nc = p->chunks.size();
    for (size_t i = 0; i < nc; ++i) {
        const auto& c = p->chunks[i];
        if (e->chunk_q_ptr) e->chunk_q_ptr[i] = qacc;
        if (e->chunk_tok_ptr) e->chunk_tok_ptr[i] = tacc;
        if (e->chunk_kind) e->chunk_kind[i] = c.kind;
        for (int32_t k = 0; k < c.dev.n_q; ++k, ++qk)
            if (e->chunk_q_mask)
                e->chunk_q_mask[qk] = c.dev.mask_base < 0 ? ~uint64_t(0) : p->masks[c.dev.mask_base + k];
        if (c.node >= 0) {
            for (int32_t t = c.tok_begin; t < c.tok_end; ++t, ++tk) {
                if (e->chunk_tok_node) e->chunk_tok_node[tk] = c.node;
                if (e->chunk_tok_t) e->chunk_tok_t[tk] = t;
            }
        } else {
            const auto& g = p->groups[p->tasks[c.task].group];
            for (size_t j = 0; j < g.tok_node.size(); ++j, ++tk) {
                if (e->chunk_tok_node) e->chunk_tok_node[tk] = g.tok_node[j];
                if (e->chunk_tok_t) e->chunk_tok_t[tk] = g.tok_t[j];
            }
        }
        qacc += c.dev.n_q;
        tacc += c.dev.n_tok;
    }
    if (e->chunk_q_ptr) e->chunk_q_ptr[nc] = qacc;
    if (e->chunk_tok_ptr) e->chunk_tok_ptr[nc] = tacc;
    return PST_OK;
}

extern "C" int pst_list_schedule(int32_t n, const double* cost, int32_t m, int32_t* slot, double* makespan) {
    if (n < 0 || m <= 0 || (n > 0 && !cost)) return fail(PST_EINVAL, "list_schedule: bad argument");
    std::vector<ItemCost> v((size_t)n);
    for (int32_t i = 0; i < n; ++i) {
        if (!(cost[i] >= 0.0)) return fail(PST_EINVAL, "list_schedule: costs must be >= 0");
        v[i] = {cost[i], i, 0, 0, 0};
    }
    std::vector<int> s;
    const double mk = list_schedule(v, m, &s);
    if (slot)
        for (int32_t k = 0; k < n; ++k) slot[v[k].chunk] = s[k];
    if (makespan) *makespan = mk;
    return PST_OK;
}
