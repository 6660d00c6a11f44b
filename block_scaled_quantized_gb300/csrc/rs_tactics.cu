// Layout autotuning (ResServe Sec. 5.1 and Fig. 3): per-shape launch tactics
// chosen by measurement instead of the planner's cost rules.
//
// A tactic fixes four choices of a linear call's plan -- the K-split count,
// in-GEMM quantization of a bf16 input, the MMA width and the weight ring
// depth of split plans -- for one
// (format, compensated, M, N, K) on a GPU with a given SM count.  The
// library ships the table measured on GB300 (rs_tactics_gb300.inc, written by
// block_scaled_quantized_gb300/tune.py, which times every candidate plan of
// each shape in CUDA graphs with the weights rotated through more than twice
// the L2 size); callers may install their own with rs_set_tactic.
//
// A call of M rows uses the entry with the smallest tuned row count >= M of
// its format, fold, N, K and SM count: within the tuned grid the plan then
// has at least the MMA width the call needs.  The planner checks that the
// tactic's plan fits (shared and tensor memory) and otherwise keeps its own.
#include <mutex>
#include <vector>

#include "rs_internal.h"

namespace rs {

namespace {

struct Entry {
    int fmt, fold, M, N, K, sms;
    Tactic t;
};

struct BuiltinRow {
    int fmt, fold, M, N, K, sms, splits, fused, bn, deep;
};

const BuiltinRow kBuiltin[] = {
#include "rs_tactics_gb300.inc"
};

std::mutex g_mu;
std::vector<Entry> g_table;
bool g_loaded = false;

bool valid(const Tactic& t) {
    return t.splits >= 1 && t.splits <= kMaxSplits && t.fused >= 0 && t.fused <= 2 &&
           (t.bn == 16 || t.bn == 32 || t.bn == 64 || t.bn == 128 || t.bn == 256) && (t.deep == 0 || t.deep == 1);
}

void put_locked(int fmt, int fold, int M, int N, int K, int sms, const Tactic& t) {
    for (Entry& e : g_table)
        if (e.fmt == fmt && e.fold == fold && e.M == M && e.N == N && e.K == K && e.sms == sms) {
            e.t = t;
            return;
        }
    g_table.push_back(Entry{fmt, fold, M, N, K, sms, t});
}

void load_builtin_locked() {
    g_table.clear();
    for (const BuiltinRow& r : kBuiltin) {
        const Tactic t{r.splits, r.fused, r.bn, r.deep};
        if (valid(t)) put_locked(r.fmt, r.fold, r.M, r.N, r.K, r.sms, t);
    }
    g_loaded = true;
}

void ensure_loaded_locked() {
    if (!g_loaded) load_builtin_locked();
}

}  // namespace

bool set_tactic(int fmt, bool fold, int M, int N, int K, int num_sms, const Tactic& t) {
    if ((fmt != 0 && fmt != 1) || M < 1 || N < 1 || K < 1 || num_sms < 1 || !valid(t)) return false;
    std::lock_guard<std::mutex> lk(g_mu);
    ensure_loaded_locked();
    put_locked(fmt, fold ? 1 : 0, M, N, K, num_sms, t);
    return true;
}

void reset_tactics(bool builtin) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (builtin) {
        load_builtin_locked();
    } else {
        g_table.clear();
        g_loaded = true;
    }
}

int tactic_count() {
    std::lock_guard<std::mutex> lk(g_mu);
    ensure_loaded_locked();
    return (int)g_table.size();
}

bool find_tactic(int fmt, bool fold, int M, int N, int K, int num_sms, Tactic* t) {
    std::lock_guard<std::mutex> lk(g_mu);
    ensure_loaded_locked();
    const Entry* best = nullptr;
    for (const Entry& e : g_table)
        if (e.fmt == fmt && e.fold == (fold ? 1 : 0) && e.N == N && e.K == K && e.sms == num_sms && e.M >= M &&
            (!best || e.M < best->M))
            best = &e;
    if (!best) return false;
    *t = best->t;
    return true;
}

}  // namespace rs
