// Shared definitions of the Gated DeltaNet kernels (warp-MMA and tcgen05 paths).
#pragma once

#include "fork_common.cuh"

namespace fork {

struct GdnParams {
  const int32_t* meta;
  MetaLayout L;
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  const float* alpha;
  const float* eta;
  const float* conv_w;      // [3, H, D, K]
  int H, K;
  const float* state_in;    // trunk: init_state (resume) or null; branch: S_P; forest: node states
  const uint16_t* hist_in;  // trunk: init_conv or null; branch: conv_win
  float* S_P;               // trunk output
  uint16_t* conv_win;       // trunk output
  float* S_ckpt;
  uint16_t* conv_ckpt;
  uint16_t* o;
  int seg_base;             // trunk call: first segment of the call (a forest level; 0 for a round)
  int n_segs;               // trunk call: its segments (-1: every trunk of the round)
  int checks;               // FORK_CHECKS
  int stall;                // FORK_TEST_STALL (tcgen05 kernel)
  uint64_t wait_ns;         // limit of a bounded wait (tcgen05 kernel)
};

// FORK_CHECKS: request j and the rows of segments [first, end) lie inside the round,
// and the segments belong to request j.
__device__ __forceinline__ bool gdn_segs_in_bounds(const int32_t* meta, const MetaLayout& L, int first, int end,
                                                   int j) {
  const int T = meta[H_T], R = meta[H_R], nseg = meta[H_NSEG];
  if (j < 0 || j >= R || first < 0 || end > nseg || end > L.max_seg) return false;
  for (int s = first; s < end; ++s) {
    const int st = meta[L.seg_start + s], len = meta[L.seg_len + s];
    if (st < 0 || len < 0 || st + len > T || meta[L.seg_req + s] != j) return false;
  }
  return true;
}

// tcgen05 kernel (d = 128); the host entry points choose between the two paths.
int launch_gdn_tc(const GdnParams& p, bool branch, int grid_x, cudaStream_t s);

}  // namespace fork
