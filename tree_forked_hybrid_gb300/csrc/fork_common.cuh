// Internal definitions shared by the CUDA sources of the ForkAttention layer.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/forkattn.h"

namespace fork {

constexpr int32_t kMagic = 0x464F524B;  // 'FORK'
constexpr int kMinTile = 8;             // smallest attention tile (Hq/Hkv = 16)

// Header words of the metadata buffer.
enum Hdr : int {
  H_MAGIC = 0, H_TCAP, H_MAXREQ, H_MAXQ, H_MAXSEG, H_MAXWORK,
  H_R, H_NQ, H_T, H_NSEG, H_TILE, H_NWORK, H_STATUS, H_PREFIX_TOTAL, H_VALID,
  H_FOREST,  // 1: the tables describe a token forest (fork_forest_plan), 0: a round
  H_WORDS = 32
};

// Offsets (in int32 words) of every metadata array; all a pure function of the
// capacities so host and device agree without reading the buffer.
struct MetaLayout {
  int32_t T_cap, max_req, max_q, max_seg, max_work;
  int64_t tok_req, tok_branch, tok_pos;
  int64_t seg_start, seg_len, seg_pos0, seg_req, seg_branch, seg_trunk_start, seg_trunk_len,
      seg_state_idx;
  int64_t req_trunk_len, req_prefix_len, req_prefix_off, req_ckpt_pos, req_trunk_start,
      req_first_q, req_n_q;
  int64_t q_last;
  int64_t work_seg, work_off, work_order;
  int64_t total;
};

__host__ __device__ inline int64_t align_words(int64_t w) { return (w + 31) & ~int64_t(31); }

__host__ __device__ inline MetaLayout meta_layout(int32_t T_cap, int32_t max_req, int32_t max_q) {
  MetaLayout L;
  L.T_cap = T_cap;
  L.max_req = max_req;
  L.max_q = max_q;
  L.max_seg = max_req + max_q;
  L.max_work = (T_cap + kMinTile - 1) / kMinTile + L.max_seg;
  int64_t o = H_WORDS;
  auto take = [&](int64_t n) { int64_t r = o; o = align_words(o + n); return r; };
  L.tok_req = take(T_cap);
  L.tok_branch = take(T_cap);
  L.tok_pos = take(T_cap);
  L.seg_start = take(L.max_seg);
  L.seg_len = take(L.max_seg);
  L.seg_pos0 = take(L.max_seg);
  L.seg_req = take(L.max_seg);
  L.seg_branch = take(L.max_seg);
  L.seg_trunk_start = take(L.max_seg);
  L.seg_trunk_len = take(L.max_seg);
  L.seg_state_idx = take(L.max_seg);
  L.req_trunk_len = take(max_req);
  L.req_prefix_len = take(max_req);
  L.req_prefix_off = take(max_req);
  L.req_ckpt_pos = take(max_req);
  L.req_trunk_start = take(max_req);
  L.req_first_q = take(max_req);
  L.req_n_q = take(max_req);
  L.q_last = take(max_q > 0 ? max_q : 1);
  L.work_seg = take(L.max_work);
  L.work_off = take(L.max_work);
  L.work_order = take(L.max_work);
  L.total = o;
  return L;
}

// Read-only view used by the compute kernels.
struct MetaView {
  const int32_t* base;
  MetaLayout L;
  __device__ __forceinline__ int32_t hdr(int i) const { return base[i]; }
  __device__ __forceinline__ int32_t at(int64_t off, int i) const { return base[off + i]; }
};

// Host: validate a caller's handle; returns FORK_OK and the layout.
int check_meta(const fork_meta* m, MetaLayout* out);

inline bool is_aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_device();  // FORK_OK on an sm_103 device, else FORK_EUNSUPPORTED/FORK_ECUDA

// Limit of the bounded waits of a call, in nanoseconds (fork_meta.wait_us; 0 = 2 s).
inline uint64_t wait_ns_of(const fork_meta* m) {
  return m->wait_us == 0 ? 2000000000ull : static_cast<uint64_t>(m->wait_us) * 1000ull;
}

// Streaming multiprocessors of the current device (grid sizing), cached per device.
int sm_count();

// Record a failing CUDA runtime result for fork_last_cuda_error (per host thread);
// returns FORK_ECUDA when e is an error, FORK_OK otherwise.
int cuda_rc(cudaError_t e);

__device__ __forceinline__ float bf2f(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}
__device__ __forceinline__ uint16_t f2bf(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}

}  // namespace fork
