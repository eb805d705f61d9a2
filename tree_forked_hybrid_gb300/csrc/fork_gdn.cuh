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
  const float* state_in;    // trunk: init_state (resume) or null; branch: S_P
  const uint16_t* hist_in;  // trunk: init_conv or null; branch: conv_win
  float* S_P;               // trunk output
  uint16_t* conv_win;       // trunk output
  float* S_ckpt;
  uint16_t* conv_ckpt;
  uint16_t* o;
};

// tcgen05 kernel (d = 128); the host entry points choose between the two paths.
int launch_gdn_tc(const GdnParams& p, bool branch, int grid_x, cudaStream_t s);

}  // namespace fork
