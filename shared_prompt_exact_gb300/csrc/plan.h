// plan.h -- packed-layout work lists shared by the host planner and the kernels.
//
// A packed micro-batch (DualKV paper, abstract: N(P+R) tokens repacked into
// P+NR) is described by P and the segment offsets.  Queries are cut into
// tiles that never cross a region boundary (the prompt, or one segment), and
// each query tile attends at most two key regions: region 0 is the shared
// prompt, region 1 the tile's own segment.  Key tiles are cut the same way.
#pragma once
#include <stdint.h>

#include <vector>

namespace dkv {

// One contiguous run of keys: rows [row0, row0+count) of the packed layout,
// with positions pos0 .. pos0+count-1.  Tiles are taken from row0 in steps of
// the kernel's key-tile size; tiles [t_lo, t_hi) hold at least one key that the
// owning query tile attends.
struct KeyRegion {
  int32_t row0, pos0, count, t_lo, t_hi;
};

// Forward / dQ work item: one query tile of one q-head.
struct QTileItem {
  int32_t q_row0;  // first packed row
  int32_t q_pos0;  // its position
  int32_t q_rows;  // valid rows (<= tile rows); rows past it belong to another region
  int32_t head;    // q-head
  KeyRegion reg[2];
};

// A block of query rows inside one region, used by the dK/dV walk.
struct QBlock {
  int32_t q_row0, q_pos0, q_rows;
};

// dK/dV work item: one key tile of one kv-head, walking iterations
// [it_lo, it_hi) of the tile's query list.  Iteration `it` is query block
// qblocks[list_begin + it / G] of group head it % G (G = Hq / Hkv): the group's
// heads of one block are consecutive.
struct KVTileItem {
  int32_t k_row0, k_pos0, k_rows, kv_head;
  int32_t list_begin, list_len;
  int32_t it_lo, it_hi;
  int32_t partial_slot;  // -1: write bf16 dk/dv directly; else fp32 partial slot
  int32_t pad_;
};

// Fixed-order reduction of split prompt key tiles.
struct ReduceItem {
  int32_t k_row0, k_rows, kv_head, slot0, nslots, pad_;
};

struct Layout {
  int P, N;
  std::vector<int32_t> off;  // N+1
  int Hq, Hkv, D, window;
  // kv-heads [kv_lo, kv_hi) and their q-head groups get work items (kv_hi < 0: all)
  int kv_lo = 0, kv_hi = -1;
  int64_t T() const { return (int64_t)P + off[N]; }
  int kv_begin() const { return kv_lo; }
  int kv_end() const { return kv_hi < 0 ? Hkv : kv_hi; }
};

// Returns an error string, or nullptr when the layout is valid.
const char* validate_layout(int P, int N, const int32_t* off, int Hq, int Hkv, int D);

// Query tiles of `tile_rows` rows and their key regions for key tiles of
// `key_tile` keys, heaviest first (by key tiles visited), ties by (head, row).
std::vector<QTileItem> plan_qtiles(const Layout& L, int tile_rows, int key_tile);

struct KVPlan {
  std::vector<KVTileItem> items;     // heaviest first
  std::vector<QBlock> qblocks;       // concatenated per-key-tile query lists
  std::vector<ReduceItem> reduces;   // one per split key tile
  int nslots = 0;                    // fp32 partial slots (each key_tile x D for dK and for dV)
};

// Key tiles of `key_tile` keys, query blocks of `q_block` rows.  A key tile
// whose walk exceeds `max_iters` iterations is split into contiguous chunks.
KVPlan plan_kvtiles(const Layout& L, int key_tile, int q_block, int max_iters);

// ---------------------------------------------------------------------------
// Head dimension 512 backward.  The 128 x 512 operand and accumulator tiles do
// not fit the fused dQ and dK/dV kernels, so the backward materialises the
// attention probabilities P and dS = P (dP - Delta) as bf16 blocks of 128 query
// rows x 128 keys in device memory, then reduces them with plain GEMMs.
// Block ids: query-tile item i (in the given list) owns blocks
// block_base[i] .. block_base[i] + (its key tiles) - 1, in walk order.
//
// One step of the dK / dV GEMM: the 64 query rows `sub` (0 or 1) of block
// `block`, i.e. rows q_row0 .. q_row0 + 63 of q-head `head`.
struct XTEntry {
  int32_t head, q_row0, block, sub;
};
// dK/dV GEMM work item: key tile x kv-head x chunk [it_lo, it_hi) of its
// entry list (group heads ascending, then query tiles in packed order).
struct XTItem {
  int32_t k_row0, k_rows, kv_head, list_begin, it_lo, it_hi, partial_slot, pad_;
};
struct Plan512 {
  std::vector<int32_t> block_base;  // per query-tile item
  int64_t n_blocks = 0;
  std::vector<XTItem> items;        // heaviest first
  std::vector<XTEntry> entries;
  std::vector<ReduceItem> reduces;
  int nslots = 0;
};
// `qitems` must come from plan_qtiles(L, 128, 128).
Plan512 plan_512(const Layout& L, const std::vector<QTileItem>& qitems, int max_iters);

// Host index builder (see dualkv_build_index).
void build_index(int P, int N, const int32_t* off, int32_t* seg_id, int32_t* pos_id, int32_t* cu_rep,
                 int32_t* rep2pack);

}  // namespace dkv
