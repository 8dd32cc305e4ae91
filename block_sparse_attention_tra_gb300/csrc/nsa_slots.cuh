// nsa_slots.cuh -- which slots of one query's block index row the NSA
// selection kernels read.
//
// Page "nsa_selection_kernel.py", selection_forward_reference: the blocks a
// query selects form a set (a one-hot scatter of the index row followed by
// `any`), so a block listed twice is read once.  A slot is live when it holds
// a block 0 <= blk < T / bs that is not wholly after the query (blk * bs <= i)
// and no earlier slot of the same row holds the same block.  Every kernel
// visits the live slots in slot order, so a producer and its consumers that
// apply this rule walk the same sequence.
#pragma once

#include <stdint.h>

namespace bsa {

// Live slots of one row, computed by a full converged warp (S <= 32): lane s
// reads slot s.  `blk_lane` is this lane's slot value (-1 for lanes >= S);
// bit s of `live` is set for every live slot s.
struct SlotRow {
  uint32_t live;
  int blk_lane;
};

__device__ __forceinline__ SlotRow nsa_live_slots(const int32_t* __restrict__ sel, int S, int i, int n_blk, int bs) {
  const int lane = static_cast<int>(threadIdx.x & 31u);
  const int blk = lane < S ? __ldg(sel + lane) : -1;
  const bool causal = blk >= 0 && blk < n_blk && blk * bs <= i;
  const uint32_t same = __match_any_sync(0xffffffffu, blk);          // lanes holding the same value
  const bool first = (same & ((1u << lane) - 1u)) == 0u;             // no earlier slot holds it
  return {__ballot_sync(0xffffffffu, causal && first), blk};
}

// Block held by slot s of a row (every lane of the warp calls it).
__device__ __forceinline__ int nsa_slot_block(const SlotRow& r, int s) {
  return __shfl_sync(0xffffffffu, r.blk_lane, s);
}

}  // namespace bsa
