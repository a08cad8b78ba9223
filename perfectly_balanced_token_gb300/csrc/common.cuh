// Internal definitions shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moonep.h"

namespace moonep {

constexpr int kMaxExperts = 4096;   // smem histograms hold E counters per warp
constexpr int kChunkCopies = 4096;  // copies per histogram chunk (rounded to tokens)
constexpr int kMmaM = 128;          // rows of one tcgen05.mma (cta_group::1)
// GEMM work-tile height, chosen before launch from the expected rows per
// weight row group, C*R/E: groups of at least this many rows use 256-row work
// tiles (two accumulators share each weight panel: fewer L2->SM bytes per
// flop); smaller groups use 128-row tiles, which keep fewer groups' weights in
// flight at once and so hit L2 more often.
constexpr int kHistWarps = 8;
// Tensor-map scratch of the grouped weight-gradient kernel: per CTA, a ring of
// kTmapSlots pairs of 128-byte tensor maps (recv and dY views whose row extent
// ends at the current group's end); sized for up to kMaxGemmCtas CTAs.
constexpr int kMaxGemmCtas = 256;
constexpr int kTmapSlots = 8;
static_assert((size_t)kMaxGemmCtas * kTmapSlots * 2 * 128 == MOONEP_GEMM_SCRATCH_BYTES,
              "the GEMM scratch at the end of the plan workspace");

// Per-expert migrated range of global ordinals [lo, hi) and where it goes.
struct Piece {
  int32_t lo, hi, u, g;
};

// One GEMM work tile of up to 128 or 256 rows (the height the plan chose): recv/y row of its first row, valid rows, the weight
// it multiplies (>= 0: home expert id; < 0: -1 - slot id u*B+j) and its rank.
struct MTile {
  int32_t row0, rows, wsel, u;
};

// Device-side view of the workspace, resolved from the layout.
struct PlanPtrs {
  int32_t* status;
  int32_t* counters;
  int32_t* counts;
  int32_t* T;
  int32_t* load;
  int32_t* keep;
  int32_t* gidx;
  int32_t* fills;
  int32_t* slot_expert;
  int32_t* n_recv;
  int32_t* src;
  int32_t* cu;
  int32_t* dst;
  int32_t* inverse;
  int32_t* route;       // [R][S][K] send-once route entries
  Piece* pieces;        // [E][R]
  int32_t* piece_n;     // [E]
  int32_t* piece_base;  // [E][R] row_base = u*C + cu[u][g] - lo
  int32_t* home_base;   // [E] home rank's row of ordinal 0 of e
  int32_t* occupied;    // [R*B]
  int32_t* red_slots;   // [E][R]
  int32_t* red_n;       // [E]
  int32_t* red_list;    // [E] experts with >= 1 slot copy
  int32_t* rank_tiles;  // [R+1] tile offset of each rank
  MTile* mtiles;        // [max_mtiles]
  int32_t* rank_groups; // [R+1] group offset of each rank
  MTile* groups;        // [max_groups] non-empty (rank, weight row) groups: all rows of each
  uint8_t* tmaps;       // [kMaxGemmCtas][kTmapSlots][2] tensor maps, 128 B each, GEMM scratch
  int32_t* sched;       // [6] work-item counters of the GEMMs, in the header the plan zeroes:
                        // {next item, finished pairs} of the pair GEMM, of the pair weight
                        // gradient, then {next item, finished CTAs} of the 128-row GEMM
};

struct Dims {
  int R, E, B, K, S, H, Hp, mode, policy;
  int L, C, N;
  int nchunk, chunk_tokens, max_mtiles, max_groups;
  int tile_m;  // GEMM work-tile height fixed by the caller (128 or 256), or 0: chosen per plan
};

// Workspace layout (host computes it; kernels receive resolved pointers).
struct Layout {
  moonep_plan_layout pub;
  size_t pieces, piece_n, piece_base, home_base, red_slots, red_n, red_list, rank_tiles,
      rank_groups, tmaps;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void set_error(int32_t* status, int32_t bit) {
  atomicOr(status, bit);
}

__device__ __forceinline__ bool plan_failed(const int32_t* status) {
  return *reinterpret_cast<const volatile int32_t*>(status) != 0;
}

}  // namespace moonep
