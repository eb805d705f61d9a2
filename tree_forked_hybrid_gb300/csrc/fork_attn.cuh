// Shared definitions of the fork-masked attention kernels.
#pragma once

#include <cuda.h>

#include "fork_common.cuh"

namespace fork {

// One contiguous key range of a query tile (see fork_attn_mma.cu).
struct KeyRange {
  const uint16_t* k;
  const uint16_t* v;
  int row0;  // first row in k/v
  int len;   // rows in the range
  int pos0;  // position of row0
};

struct AttnParams {
  const int32_t* meta;
  MetaLayout L;
  const uint16_t* q;         // [T_cap, Hq, d]
  const uint16_t* k;         // stream keys [T_cap, Hkv, d] (rotated copy when rope is on)
  const uint16_t* v;         // [T_cap, Hkv, d]
  const uint16_t* prefix_k;  // [prefix_rows, Hkv, d] (rotated copy when rope is on)
  const uint16_t* prefix_v;
  uint16_t* o;
  const float2* rope_hi;     // (cos, sin) of 64*a*f_i, [a][d/2]
  const float2* rope_lo;     // (cos, sin) of b*f_i,    [b < 64][d/2]
  int Hq, Hkv, G;
  int prefix_rows;           // rows of prefix_k / prefix_v
  int window;
  float rope_theta;          // 0 = off
  float scale_log2;          // scale * log2(e)
  int rope_hi_rows;          // rows of rope_hi
  int rotate_q;              // queries are rotated by the attention kernel (tcgen05 path)
  int checks;                // FORK_CHECKS
  int stall;                 // FORK_TEST_STALL (tcgen05 path)
  uint64_t wait_ns;          // limit of a bounded wait
  int* work_ctr;             // tcgen05 path: work items claimed so far (zeroed before the kernel)
};

// FORK_CHECKS: work item w's segment, its offset, its request and its trunk range lie
// inside the round (the prefix range is checked against the prefix buffers separately).
__device__ __forceinline__ bool attn_item_in_bounds(const int32_t* meta, const MetaLayout& L, int w) {
  const int T = meta[H_T], nseg = meta[H_NSEG], R = meta[H_R];
  if (meta[H_NWORK] > L.max_work || w < 0 || w >= meta[H_NWORK]) return false;
  const int s = meta[L.work_seg + w];
  if (s < 0 || s >= nseg || s >= L.max_seg) return false;
  const int st = meta[L.seg_start + s], len = meta[L.seg_len + s], off = meta[L.work_off + w];
  const int j = meta[L.seg_req + s];
  const int ts = meta[L.seg_trunk_start + s], tl = meta[L.seg_trunk_len + s];
  return st >= 0 && len >= 1 && st + len <= T && off >= 0 && off < len && j >= 0 && j < R && ts >= 0 &&
         tl >= 0 && ts + tl <= T;
}

// (cos, sin) of t * f_i from the two-level table: t = 64 a + b,
// angle(t) = angle(64 a) + angle(b), combined by the angle-addition formula.
__device__ __forceinline__ void rope_cs(const float2* hi, const float2* lo, int half, int t, int i,
                                        float* cs, float* sn) {
  const float2 A = hi[(t >> 6) * half + i];
  const float2 B = lo[(t & 63) * half + i];
  *cs = A.x * B.x - A.y * B.y;
  *sn = A.y * B.x + A.x * B.y;
}

// TMA descriptor of a bf16 tensor [rows][heads][d] (fork_attn.cu)
bool encode_map_3d(CUtensorMap* m, const void* base, int d, int heads, int64_t rows, int box_d, int box_heads,
                   int box_rows, bool swizzle128);

template <int D>
int launch_attn_mma(const AttnParams& p, int grid_x, cudaStream_t s);

// maps: q, k, v, prefix k, prefix v (CUtensorMap, 128-byte aligned); forest: the metadata
// describes a token forest (D = 128)
template <int D>
int launch_attn_tc(const AttnParams& p, const CUtensorMap* maps, int grid_x, bool two_tiles, bool forest,
                   cudaStream_t s);

}  // namespace fork
