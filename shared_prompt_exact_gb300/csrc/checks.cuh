// checks.cuh -- device-side range checks of work-list entries.
//
// Every row a kernel reads or writes is derived from its work list, which the
// host planner builds inside the tensors.  These predicates confirm that
// before any access: a kernel that finds an entry outside the tensors records
// kDevErrBounds in the status word (dualkv_check_status reports it) and skips
// the entry's loads and stores, so a corrupted list cannot become a memory fault.
#pragma once
#include <stdint.h>

#include "plan.h"

namespace dkv {

__device__ __forceinline__ bool rows_ok(int64_t row0, int64_t rows, int64_t T, int max_rows) {
  return row0 >= 0 && rows >= 0 && rows <= max_rows && row0 + rows <= T;
}

// A key region of a query-tile item: its rows lie in [0, T) and its tile range
// [t_lo, t_hi) lies inside ceil(count / key_tile) tiles.
__device__ __forceinline__ bool region_ok(const KeyRegion& r, int64_t T, int key_tile) {
  if (r.t_lo == r.t_hi) return r.t_lo >= 0;
  // t_hi <= ceil(count / key_tile), without a division
  return r.row0 >= 0 && r.count >= 0 && (int64_t)r.row0 + r.count <= T && r.t_lo >= 0 && r.t_lo < r.t_hi &&
         (int64_t)(r.t_hi - 1) * key_tile < (int64_t)r.count;
}

// A forward / dQ / D = 512 block work item: query tile of at most tile_rows rows of
// q-head `head`, and its two key regions.
__device__ __forceinline__ bool qtile_ok(const QTileItem& it, int64_t T, int Hq, int tile_rows, int key_tile) {
  return rows_ok(it.q_row0, it.q_rows, T, tile_rows) && it.head >= 0 && it.head < Hq &&
         region_ok(it.reg[0], T, key_tile) && region_ok(it.reg[1], T, key_tile);
}

}  // namespace dkv
