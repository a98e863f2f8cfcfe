// Host control plane: see host_plan.h.
#include "host_plan.h"

#include <algorithm>
#include <climits>

namespace llm {

// ---------------------------------------------------------------------------------------------
// llama_batch_allocr::init ([P1] Крок 10): checks, then defaults for the fields left NULL.
bool sanitize_batch(int32_t n, const int32_t* token, const int32_t* pos, const int32_t* n_seq_id,
                    const int32_t* const* seq_id, const int8_t* logits, int32_t n_vocab,
                    int32_t n_seq_max, int32_t n_batch, const KvCells& cells, SanBatch& out,
                    std::string* why) {
    auto fail = [&](const std::string& m) { if (why) *why = m; return false; };
    if (n <= 0) return fail("batch has no tokens");
    if (n > n_batch) return fail("batch has more than n_batch tokens");
    if (!token) return fail("batch token array is NULL (embeddings input is not supported)");
    out.n = n;
    out.token.assign(token, token + n);
    for (int32_t i = 0; i < n; ++i)
        if (token[i] < 0 || token[i] >= n_vocab) return fail("token id out of range");
    out.seqs.assign(n, SeqSet());
    out.first_seq.assign(n, 0);
    for (int32_t i = 0; i < n; ++i) {
        if (!seq_id) { out.seqs[i].set(0); continue; }
        const int32_t k = n_seq_id ? n_seq_id[i] : 1;
        if (k < 1 || k > kMaxSeq) return fail("n_seq_id out of range");
        if (!seq_id[i]) return fail("seq_id row is NULL");
        for (int32_t j = 0; j < k; ++j) {
            const int32_t s = seq_id[i][j];
            if (s < 0 || s >= n_seq_max) return fail("sequence id out of range");
            out.seqs[i].set(s);
        }
        out.first_seq[i] = seq_id[i][0];
    }
    // positions: continue each sequence from the memory, in batch order
    out.pos.assign(n, 0);
    std::vector<int32_t> next(n_seq_max, INT_MIN);
    auto start_of = [&](int32_t s) {
        if (next[s] == INT_MIN) next[s] = cells.seq_pos_max(s) + 1;
        return next[s];
    };
    if (!pos) {
        for (int32_t i = 0; i < n; ++i) {
            const int32_t p = start_of(out.first_seq[i]);
            out.pos[i] = p;
            for (int32_t s = 0; s < n_seq_max; ++s)
                if (out.seqs[i].test(s)) next[s] = p + 1;
        }
    } else {
        out.pos.assign(pos, pos + n);
    }
    // consistency: each sequence's positions are consecutive and continue from seq_pos_max + 1
    std::vector<int32_t> last(n_seq_max, INT_MIN);
    for (int32_t i = 0; i < n; ++i) {
        for (int32_t s = 0; s < n_seq_max; ++s) {
            if (!out.seqs[i].test(s)) continue;
            const int32_t want = last[s] == INT_MIN ? cells.seq_pos_max(s) + 1 : last[s] + 1;
            if (out.pos[i] != want) return fail("positions of a sequence are not consecutive");
            last[s] = out.pos[i];
        }
    }
    out.output.assign(n, 0);
    if (!logits) out.output[n - 1] = 1;
    else for (int32_t i = 0; i < n; ++i) out.output[i] = logits[i] != 0;
    out.n_outputs = 0;
    for (int32_t i = 0; i < n; ++i) out.n_outputs += out.output[i];
    return true;
}

// ---------------------------------------------------------------------------------------------
KvCells::KvCells(int32_t n_ctx, int32_t n_seq_max, int32_t n_stream)
    : pos_(n_ctx, -1), seq_(n_ctx), seq_pos_(n_seq_max), sc_(n_seq_max), sp_(n_seq_max),
      n_stream_(n_stream < 1 ? 1 : n_stream), n_ctx_seq_(n_ctx / (n_stream < 1 ? 1 : n_stream)) {
    free_lo_.resize(n_stream_);
    for (int32_t s = 0; s < n_stream_; ++s) free_lo_[s] = stream_lo(s);
}

int32_t KvCells::seq_pos_max(int32_t s) const {
    if (s < 0 || s >= (int32_t)seq_pos_.size() || seq_pos_[s].empty()) return -1;
    return seq_pos_[s].rbegin()->first;
}

int32_t KvCells::seq_pos_min(int32_t s) const {
    if (s < 0 || s >= (int32_t)seq_pos_.size() || seq_pos_[s].empty()) return -1;
    return seq_pos_[s].begin()->first;
}

bool KvCells::find_free(int32_t n, std::vector<int32_t>& out, int32_t stream) const {
    out.clear();
    if (stream < 0 || stream >= n_stream_) return n == 0;
    const int32_t hi = stream_hi(stream);
    for (int32_t c = free_lo_[stream]; c < hi && (int32_t)out.size() < n; ++c)
        if (pos_[c] < 0) out.push_back(c);
    return (int32_t)out.size() == n;
}

void KvCells::apply(const std::vector<int32_t>& slots, const int32_t* pos, const SeqSet* seqs,
                    int32_t n) {
    const int32_t ns = (int32_t)seq_pos_.size();
    for (int32_t i = 0; i < n; ++i) {
        const int32_t c = slots[i];
        pos_[c] = pos[i];
        seq_[c] = seqs[i];
        for (int32_t s = 0; s < ns; ++s) {
            if (!seqs[i].test(s)) continue;
            seq_pos_[s][pos[i]] += 1;
            auto& cs = sc_[s];
            auto& ps = sp_[s];
            if (cs.empty() || cs.back() < c) {
                cs.push_back(c);
                ps.push_back(pos[i]);
            } else {
                const auto it = std::lower_bound(cs.begin(), cs.end(), c);
                const auto k = it - cs.begin();
                cs.insert(it, c);
                ps.insert(ps.begin() + k, pos[i]);
            }
        }
        used_ += 1;
        used_max_ = std::max(used_max_, c);
    }
    for (int32_t s = 0; s < n_stream_; ++s)
        while (free_lo_[s] < stream_hi(s) && pos_[free_lo_[s]] >= 0) ++free_lo_[s];
}

void KvCells::free_cell(int32_t c) {
    pos_[c] = -1;
    used_ -= 1;
    const int32_t s = std::min(stream_of(c), n_stream_ - 1);
    free_lo_[s] = std::min(free_lo_[s], c);
    while (used_max_ >= 0 && pos_[used_max_] < 0) --used_max_;
}

void KvCells::drop_seq_from_cell(int32_t c, int32_t s) {
    seq_[c].reset(s);
    auto it = seq_pos_[s].find(pos_[c]);
    if (it != seq_pos_[s].end() && --(it->second) == 0) seq_pos_[s].erase(it);
    auto& cs = sc_[s];
    const auto jt = std::lower_bound(cs.begin(), cs.end(), c);
    if (jt != cs.end() && *jt == c) {
        const auto k = jt - cs.begin();
        cs.erase(jt);
        sp_[s].erase(sp_[s].begin() + k);
    }
    if (seq_[c].none()) free_cell(c);
}

void KvCells::seq_rm(int32_t s, int32_t p0, int32_t p1) {
    if (p0 < 0) p0 = 0;
    if (p1 < 0) p1 = INT_MAX;
    const int32_t ns = (int32_t)seq_pos_.size();
    for (int32_t q = (s < 0 ? 0 : s); q < (s < 0 ? ns : std::min(s + 1, ns)); ++q) {
        std::vector<int32_t> victims;
        const auto& cs = sc_[q];
        const auto& ps = sp_[q];
        for (size_t k = 0; k < cs.size(); ++k)
            if (ps[k] >= p0 && ps[k] < p1) victims.push_back(cs[k]);
        for (int32_t c : victims) drop_seq_from_cell(c, q);
    }
}

bool KvCells::defrag_order(std::vector<int32_t>& src) const {
    struct Key { int32_t seq, pos, cell; };
    src.assign(size(), -1);
    bool moved = false;
    std::vector<Key> keys;
    for (int32_t st = 0; st < n_stream_; ++st) {
        keys.clear();
        const int32_t lo = stream_lo(st), hi = stream_hi(st);
        for (int32_t cl = lo; cl < hi; ++cl) {
            if (pos_[cl] < 0) continue;
            int32_t s = 0;
            while (s < kMaxSeq && !seq_[cl].test(s)) ++s;
            keys.push_back({s, pos_[cl], cl});
        }
        std::sort(keys.begin(), keys.end(), [](const Key& a, const Key& b) {
            if (a.seq != b.seq) return a.seq < b.seq;
            if (a.pos != b.pos) return a.pos < b.pos;
            return a.cell < b.cell;
        });
        for (size_t i = 0; i < keys.size(); ++i) {
            src[lo + i] = keys[i].cell;
            moved = moved || keys[i].cell != lo + (int32_t)i;
        }
    }
    return moved;
}

void KvCells::move(const std::vector<int32_t>& src) {
    KvCells fresh(size(), (int32_t)seq_pos_.size(), n_stream_);
    std::vector<int32_t> slot(1), p(1);
    for (int32_t i = 0; i < (int32_t)src.size(); ++i) {
        if (src[i] < 0) continue;
        slot[0] = i;
        p[0] = pos_[src[i]];
        fresh.apply(slot, p.data(), &seq_[src[i]], 1);
    }
    *this = std::move(fresh);
}

void split_equal(const std::vector<int32_t>& seq_of, int32_t n_ubatch, std::vector<int32_t>& order,
                 std::vector<int32_t>& ub_off) {
    std::map<int32_t, std::vector<int32_t>> queues;           // ascending sequence id
    for (int32_t i = 0; i < (int32_t)seq_of.size(); ++i) queues[seq_of[i]].push_back(i);
    std::map<int32_t, size_t> head;
    order.clear();
    ub_off.assign(1, 0);
    std::vector<int32_t> sets;
    while (true) {
        sets.clear();
        for (const auto& q : queues) {
            if (head[q.first] >= q.second.size()) continue;
            if (!sets.empty() && (q.first != sets.back() + 1 || (int32_t)sets.size() >= n_ubatch)) break;
            sets.push_back(q.first);
        }
        if (sets.empty()) return;
        size_t n_seq_tokens = (size_t)(n_ubatch / (int32_t)sets.size());
        for (int32_t s : sets) n_seq_tokens = std::min(n_seq_tokens, queues[s].size() - head[s]);
        for (int32_t s : sets) {
            const auto& q = queues[s];
            for (size_t k = 0; k < n_seq_tokens; ++k) order.push_back(q[head[s] + k]);
            head[s] += n_seq_tokens;
        }
        ub_off.push_back((int32_t)order.size());
    }
}

// ---------------------------------------------------------------------------------------------
void build_attn_plan(const KvCells& cells, const SanBatch& b, int32_t i0, int32_t T, int32_t tile_q,
                     int32_t n_head_kv, int32_t n_gqa, int32_t target_items, int32_t max_rows,
                     int32_t max_work, AttnPlan& p, int32_t min_chunk) {
    p.list_off.assign(1, 0);
    p.list_cells.clear();
    p.list_pos.clear();
    p.tok_list.assign(T, -1);
    std::vector<SeqSet> sets;
    std::vector<int32_t> single(kMaxSeq, -1);
    for (int32_t t = 0; t < T; ++t) {
        const SeqSet& ss = b.seqs[i0 + t];
        int32_t id = -1;
        if (ss.count() == 1) {
            id = single[b.first_seq[i0 + t]];
        } else {
            for (size_t j = 0; j < sets.size(); ++j)
                if (sets[j] == ss) { id = (int32_t)j; break; }
        }
        if (id < 0) {
            id = (int32_t)sets.size();
            sets.push_back(ss);
            if (ss.count() == 1) single[b.first_seq[i0 + t]] = id;
            // the list: cells sharing a sequence with the set, ascending
            if (ss.count() == 1) {
                const int32_t s = b.first_seq[i0 + t];
                p.list_cells.insert(p.list_cells.end(), cells.seq_cells(s).begin(), cells.seq_cells(s).end());
                p.list_pos.insert(p.list_pos.end(), cells.seq_cell_pos(s).begin(), cells.seq_cell_pos(s).end());
            } else {
                std::vector<std::pair<int32_t, int32_t>> u;
                for (int32_t s = 0; s < kMaxSeq; ++s) {
                    if (!ss.test(s)) continue;
                    const auto& cs = cells.seq_cells(s);
                    const auto& ps = cells.seq_cell_pos(s);
                    for (size_t k = 0; k < cs.size(); ++k) u.emplace_back(cs[k], ps[k]);
                }
                std::sort(u.begin(), u.end());
                u.erase(std::unique(u.begin(), u.end()), u.end());
                for (auto& e : u) { p.list_cells.push_back(e.first); p.list_pos.push_back(e.second); }
            }
            p.list_off.push_back((int32_t)p.list_cells.size());
        }
        p.tok_list[t] = id;
    }
    const int32_t nl = (int32_t)sets.size();
    // group tokens by list, cut into query tiles
    p.perm.clear();
    p.tile_list.clear(); p.tile_start.clear(); p.tile_nq.clear();
    p.tok_tile.assign(T, 0); p.tok_row.assign(T, 0);
    p.max_nq = 0;
    std::vector<std::vector<int32_t>> members(nl);
    for (int32_t t = 0; t < T; ++t) members[p.tok_list[t]].push_back(t);
    for (int32_t l = 0; l < nl; ++l) {
        for (size_t k = 0; k < members[l].size(); k += tile_q) {
            const int32_t nq = (int32_t)std::min<size_t>(tile_q, members[l].size() - k);
            const int32_t tile = (int32_t)p.tile_list.size();
            p.tile_list.push_back(l);
            p.tile_start.push_back((int32_t)p.perm.size());
            p.tile_nq.push_back(nq);
            p.max_nq = std::max(p.max_nq, nq);
            for (int32_t j = 0; j < nq; ++j) {
                const int32_t t = members[l][k + j];
                p.perm.push_back(t);
                p.tok_tile[t] = tile;
                p.tok_row[t] = j;
            }
        }
    }
    // split each tile's list into work items; list entries past the last one any token of the
    // tile may see (position <= the tile's largest position) are left out
    const int32_t nt = (int32_t)p.tile_list.size();
    std::vector<int32_t> tile_len(nt);
    for (int32_t t = 0; t < nt; ++t) {
        const int32_t l = p.tile_list[t];
        int32_t pmax = INT32_MIN;
        for (int32_t j = 0; j < p.tile_nq[t]; ++j) pmax = std::max(pmax, b.pos[i0 + p.perm[p.tile_start[t] + j]]);
        int32_t L = p.list_off[l + 1] - p.list_off[l];
        while (L > 1 && p.list_pos[p.list_off[l] + L - 1] > pmax) --L;
        tile_len[t] = L;
    }
    int32_t want = std::max(1, target_items / std::max(1, nt * n_head_kv));
    for (;;) {
        p.wi_tile.clear(); p.wi_c0.clear(); p.wi_c1.clear();
        p.wi_row_off.assign(1, 0);
        p.tile_wi_off.assign(1, 0);
        for (int32_t t = 0; t < nt; ++t) {
            const int32_t L = tile_len[t];
            int32_t chunk = (L + want - 1) / want;
            const int32_t gran = std::min<int32_t>(32, min_chunk);
            chunk = std::max(min_chunk, (chunk + gran - 1) / gran * gran);
            for (int32_t c0 = 0; c0 < std::max(L, 1); c0 += chunk) {
                p.wi_tile.push_back(t);
                p.wi_c0.push_back(c0);
                p.wi_c1.push_back(std::min(L, c0 + chunk));
                p.wi_row_off.push_back(p.wi_row_off.back() + p.tile_nq[t] * n_gqa);
            }
            p.tile_wi_off.push_back((int32_t)p.wi_tile.size());
        }
        if ((p.wi_row_off.back() <= max_rows && (int32_t)p.wi_tile.size() <= max_work) || want == 1)
            break;
        want = std::max(1, want / 2);
    }
}

}  // namespace llm
