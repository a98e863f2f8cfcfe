// Host control plane of the decode path: batch sanitising, ubatch split, KV cells, slot search,
// and the per-ubatch attention plan (which cached cells each token may read).
//
// [P1] "llama.cpp AI LLM Engine - Як це працює", Крок 10 (llama_batch_allocr::init), Крок 12
// (llama_kv_cache::init_batch), Крок 13а (mctx->apply); [P4] "デコードループ" KVキャッシュの詳細
// (llama_kv_cells: pos, seq bitset, per-sequence positions) and エラーリカバリ (seq_rm rollback).
#pragma once

#include <bitset>
#include <cstdint>
#include <map>
#include <string>
#include <vector>

namespace llm {

constexpr int kMaxSeq = 256;            // sequence ids are 0 .. n_seq_max-1, n_seq_max <= 256
using SeqSet = std::bitset<kMaxSeq>;

// A batch after sanitising: every field filled in.
struct SanBatch {
    int32_t n = 0;
    std::vector<int32_t> token, pos;
    std::vector<SeqSet> seqs;
    std::vector<int32_t> first_seq;      // seq_id[i][0]
    std::vector<uint8_t> output;
    int32_t n_outputs = 0;
};

class KvCells;

// llama_batch_allocr::init: validate and fill defaults. Returns false for an invalid batch
// (the caller turns that into -1) and sets *why.
bool sanitize_batch(int32_t n_tokens, const int32_t* token, const int32_t* pos,
                    const int32_t* n_seq_id, const int32_t* const* seq_id, const int8_t* logits,
                    int32_t n_vocab, int32_t n_seq_max, int32_t n_batch, const KvCells& cells,
                    SanBatch& out, std::string* why);

// The cells of the cache. A cell holds one position (-1 = empty) and the set of sequences that
// use it. Per sequence the library keeps its cells sorted by index (with their positions), which
// is what the attention plan reads. n_stream > 1: a cache not shared by all sequences ([P1] Крок
// 9-10, n_ctx divided among the sequences): stream s owns cells [s n_ctx_seq, (s + 1) n_ctx_seq),
// n_ctx_seq = n_ctx / n_stream, and a token's cells come from its sequence's stream.
class KvCells {
public:
    explicit KvCells(int32_t n_ctx = 0, int32_t n_seq_max = 1, int32_t n_stream = 1);

    int32_t n_stream() const { return n_stream_; }
    int32_t n_ctx_seq() const { return n_ctx_seq_; }

    int32_t size() const { return (int32_t)pos_.size(); }
    int32_t used() const { return used_; }
    int32_t n_kv() const { return used_max_ + 1; }   // highest used cell + 1
    int32_t pos(int32_t c) const { return pos_[c]; }
    const SeqSet& seqs(int32_t c) const { return seq_[c]; }

    int32_t seq_pos_max(int32_t s) const;
    int32_t seq_pos_min(int32_t s) const;

    // Cells of sequence s sorted by cell index, and their positions (parallel arrays).
    const std::vector<int32_t>& seq_cells(int32_t s) const { return sc_[s]; }
    const std::vector<int32_t>& seq_cell_pos(int32_t s) const { return sp_[s]; }

    // The n lowest-index empty cells of a stream, ascending, without claiming them. False if
    // fewer are empty.
    bool find_free(int32_t n, std::vector<int32_t>& out, int32_t stream = 0) const;

    // Commit tokens to cells (mctx->apply). Cells must be empty.
    void apply(const std::vector<int32_t>& slots, const int32_t* pos, const SeqSet* seqs, int32_t n);

    // Remove sequence s (s < 0: every sequence) from cells with p0 <= pos < p1 (p0 < 0 -> 0,
    // p1 < 0 -> no bound). A cell left with no sequence becomes empty.
    void seq_rm(int32_t s, int32_t p0, int32_t p1);

    // Defrag ([P4] KVキャッシュの詳細, memory_update(optimize=true) and its "After Defrag"
    // figure): in each stream the used cells packed from the stream's first cell, ordered by
    // their lowest sequence id, then position, then cell. src[i] (size n_ctx) = the old cell that
    // cell i takes, -1 = empty. False if no cell moves.
    bool defrag_order(std::vector<int32_t>& src) const;
    // Rewrite the cells so that cell i holds what old cell src[i] held (-1: empty).
    void move(const std::vector<int32_t>& src);

private:
    void drop_seq_from_cell(int32_t c, int32_t s);
    void free_cell(int32_t c);

    std::vector<int32_t> pos_;
    std::vector<SeqSet> seq_;
    std::vector<std::map<int32_t, int32_t>> seq_pos_;   // per sequence: position -> cell count
    std::vector<std::vector<int32_t>> sc_, sp_;         // per sequence: sorted cells, their pos
    int32_t used_ = 0;
    int32_t used_max_ = -1;
    int32_t n_stream_ = 1, n_ctx_seq_ = 0;
    std::vector<int32_t> free_lo_;                      // per stream: its cells below are used
    int32_t stream_lo(int32_t s) const { return n_stream_ == 1 ? 0 : s * n_ctx_seq_; }
    int32_t stream_hi(int32_t s) const { return n_stream_ == 1 ? size() : (s + 1) * n_ctx_seq_; }
    int32_t stream_of(int32_t c) const { return n_stream_ == 1 ? 0 : c / n_ctx_seq_; }
};

// split_equal(n_ubatch, sequential = true) ([P1] Крок 12: the splitter of a cache with more than
// one stream; [P4] llama_ubatch: n_seq_tokens tokens per sequence set, n_seqs sets). Every token
// has one sequence (seq_of). A ubatch takes the sequences with unused tokens in ascending id,
// consecutive ids only, at most n_ubatch of them; each gives n_seq_tokens = min(n_ubatch /
// n_seqs, fewest unused tokens among them) of its next tokens in batch order, listed sequence by
// sequence. order = batch indices in ubatch order; ub_off = ubatch boundaries in order (n_ub + 1).
void split_equal(const std::vector<int32_t>& seq_of, int32_t n_ubatch, std::vector<int32_t>& order,
                 std::vector<int32_t>& ub_off);

// Attention plan of one ubatch, after its cells are committed.
//  - A "list" is the ascending set of cells shared with one distinct sequence set of the ubatch's
//    tokens; a token may read a cell of its list iff cell.pos <= token.pos (causal).
//  - Tokens are grouped by list (perm) and cut into query tiles of at most tile_q tokens.
//  - Each tile's list is cut into work items of at most chunk cells (split-K over the cache); list
//    entries after the last one with a position <= the tile's largest token position are left out
//    (no token of the tile may see them).
struct AttnPlan {
    std::vector<int32_t> list_off;      // [n_lists + 1]
    std::vector<int32_t> list_cells;    // concatenated cell indices
    std::vector<int32_t> list_pos;      // their positions
    std::vector<int32_t> tok_list;      // [T] list of each token
    std::vector<int32_t> perm;          // [T] token indices grouped by list
    std::vector<int32_t> tile_list, tile_start, tile_nq;   // per query tile
    std::vector<int32_t> wi_tile, wi_c0, wi_c1;            // per work item (cell range in list)
    std::vector<int32_t> wi_row_off;    // [n_work + 1] first partial-result row of each work item
    std::vector<int32_t> tile_wi_off;   // [n_tiles + 1] work items of each tile
    std::vector<int32_t> tok_tile, tok_row;                // [T] tile of a token and its row in it
    int32_t max_nq = 0;
    int32_t n_lists() const { return (int32_t)list_off.size() - 1; }
    int32_t n_tiles() const { return (int32_t)tile_list.size(); }
    int32_t n_work() const { return (int32_t)wi_tile.size(); }
};

// Build the plan for ubatch tokens [i0, i0 + T) of a sanitised batch. target_items is the number
// of (work item x KV head) blocks the split aims for; chunk sizes are multiples of 32 cells. A work
// item of a tile with nq tokens produces nq * n_gqa partial rows; the split is coarsened until
// the rows of all work items fit in max_rows and the items in max_work (one item per tile
// always fits when max_rows >= T * n_gqa and max_work >= T).
void build_attn_plan(const KvCells& cells, const SanBatch& b, int32_t i0, int32_t T,
                     int32_t tile_q, int32_t n_head_kv, int32_t n_gqa, int32_t target_items,
                     int32_t max_rows, int32_t max_work, AttnPlan& plan, int32_t min_chunk = 32);

}  // namespace llm
