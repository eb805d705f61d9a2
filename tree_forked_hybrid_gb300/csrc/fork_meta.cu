// Round metadata builder: per-token (j, c, t), segment and request tables,
// question last rows and the attention work list, built on the device from
// the packed round descriptor.
//
// Source: Flide pages - onedev summary "무엇과 다른가" (flat unpadded stream
// [s(1)|s(2)|...|q1(1)|...], per-token request/branch/position, question
// positions continue from P) and "어떻게 쓰나" (segment lengths, positions,
// key ranges and state indices held in device buffers, kernels size their
// work from them); rainbus summary "方法步骤详情" steps 1 and 3.
#include <cstdio>

#include "fork_common.cuh"

namespace fork {

static thread_local int t_last_cuda_error = 0;
constexpr int kSortMax = 4096;  // work lists up to this length are launched longest first

int cuda_rc(cudaError_t e) {
  if (e == cudaSuccess) return FORK_OK;
  t_last_cuda_error = static_cast<int>(e);
  return FORK_ECUDA;
}

int check_device() {
  int dev = 0;
  if (cuda_rc(cudaGetDevice(&dev)) != FORK_OK) return FORK_ECUDA;
  int major = 0, minor = 0;
  if (cuda_rc(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != FORK_OK ||
      cuda_rc(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != FORK_OK)
    return FORK_ECUDA;
  return (major == 10 && minor == 3) ? FORK_OK : FORK_EUNSUPPORTED;
}

int sm_count() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) return 1;
    cached[dev] = n;
  }
  return cached[dev];
}

static bool valid_caps(int32_t T_cap, int32_t max_req, int32_t max_q) {
  return T_cap >= 1 && T_cap <= (1 << 20) && max_req >= 1 && max_req <= (1 << 16) && max_q >= 0 &&
         max_q <= (1 << 18);
}

int check_meta(const fork_meta* m, MetaLayout* out) {
  if (!m || !m->d_buf || !is_aligned16(m->d_buf)) return FORK_EINVAL;
  if (!valid_caps(m->T_cap, m->max_req, m->max_q)) return FORK_EINVAL;
  int t = m->tile_tokens;
  if (t != 8 && t != 16 && t != 32 && t != 64 && t != 128 && t != 256) return FORK_EINVAL;
  MetaLayout L = meta_layout(m->T_cap, m->max_req, m->max_q);
  if (m->bytes < static_cast<size_t>(L.total) * 4) return FORK_EINVAL;
  *out = L;
  return FORK_OK;
}

// Block-wide exclusive prefix sum over n values produced by val(i); store(i, prefix)
// receives each exclusive prefix.  Returns the total to every thread.
template <typename F, typename G>
__device__ long long block_scan(int n, F val, G store) {
  __shared__ long long warp_sums[32];
  __shared__ long long carry;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < n; base += blockDim.x) {
    const int i = base + threadIdx.x;
    const long long v = (i < n) ? static_cast<long long>(val(i)) : 0;
    long long x = v;
    for (int o = 1; o < 32; o <<= 1) {
      long long y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
      long long w = (lane < nwarps) ? warp_sums[lane] : 0;
      for (int o = 1; o < 32; o <<= 1) {
        long long y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      warp_sums[lane] = w;
    }
    __syncthreads();
    const long long excl = carry + (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
    if (i < n) store(i, excl);
    __syncthreads();
    if (threadIdx.x == 0) carry += warp_sums[nwarps - 1];
    __syncthreads();
  }
  return carry;
}

// One block: validation, request and segment tables, question rows, work list.
// dev_counts = 0: desc = [R P | R n | Nq q_len | R prefix | R ckpt] with R, Nq given;
// dev_counts = 1: desc = [R, Nq | max_req P | max_req n | max_q q_len | max_req prefix |
// max_req ckpt], the counts read here (nothing on the host depends on them).
__global__ void __launch_bounds__(1024) meta_tables_kernel(const int32_t* __restrict__ desc, int R,
                                                           int Nq, int dev_counts, int32_t* __restrict__ meta,
                                                           MetaLayout L, int tile) {
  __shared__ int s_bad;
  if (threadIdx.x == 0) s_bad = 0;
  const int32_t *P, *n, *ql, *pl, *ck;
  int over = 0;
  if (dev_counts) {
    R = desc[0];
    Nq = desc[1];
    over = (R < 0 || R > L.max_req || Nq < 0 || Nq > L.max_q) ? 1 : 0;
    if (over) R = Nq = 0;
    P = desc + 2;
    n = P + L.max_req;
    ql = n + L.max_req;
    pl = ql + L.max_q;
    ck = pl + L.max_req;
  } else {
    P = desc;
    n = desc + R;
    ql = desc + 2 * R;
    pl = desc + 2 * R + Nq;
    ck = desc + 3 * R + Nq;
  }
  __syncthreads();
  if (over && threadIdx.x == 0) s_bad = FORK_STATUS_CAPACITY;

  // ---- validation --------------------------------------------------------
  int bad = 0;
  for (int j = threadIdx.x; j < R; j += blockDim.x) {
    const int32_t Pj = P[j], nj = n[j], plj = pl[j], ckj = ck[j];
    if (Pj < 0 || nj < 0 || plj < 0 || plj > Pj) bad |= FORK_STATUS_BAD_DESC;
    if (ckj != -1 && (ckj < plj || ckj > Pj)) bad |= FORK_STATUS_BAD_CKPT;
  }
  for (int i = threadIdx.x; i < Nq; i += blockDim.x)
    if (ql[i] < 1) bad |= FORK_STATUS_BAD_DESC;
  if (bad) atomicOr(&s_bad, bad);
  __syncthreads();
  long long sum_n = block_scan(R, [&](int j) { return n[j] < 0 ? 0 : n[j]; }, [](int, long long) {});
  long long T_trunk = block_scan(
      R, [&](int j) { return (P[j] >= pl[j] && pl[j] >= 0) ? P[j] - pl[j] : 0; }, [](int, long long) {});
  long long T_q = block_scan(Nq, [&](int i) { return ql[i] < 0 ? 0 : ql[i]; }, [](int, long long) {});
  if (threadIdx.x == 0) {
    if (sum_n != Nq) s_bad |= FORK_STATUS_BAD_DESC;
    if (T_trunk + T_q > L.T_cap) s_bad |= FORK_STATUS_CAPACITY;
  }
  __syncthreads();
  const int status = s_bad;
  if (threadIdx.x == 0) {
    meta[H_MAGIC] = kMagic;
    meta[H_TCAP] = L.T_cap;
    meta[H_MAXREQ] = L.max_req;
    meta[H_MAXQ] = L.max_q;
    meta[H_MAXSEG] = L.max_seg;
    meta[H_MAXWORK] = L.max_work;
    meta[H_R] = status ? 0 : R;
    meta[H_NQ] = status ? 0 : Nq;
    meta[H_T] = status ? 0 : static_cast<int32_t>(T_trunk + T_q);
    meta[H_NSEG] = status ? 0 : R + Nq;
    meta[H_TILE] = tile;
    meta[H_STATUS] = status;
    meta[H_VALID] = status ? 0 : 1;
    meta[H_FOREST] = 0;
  }
  if (status) {
    if (threadIdx.x == 0) {
      meta[H_NWORK] = 0;
      meta[H_PREFIX_TOTAL] = 0;
    }
    return;
  }

  // ---- request table ----------------------------------------------------
  int32_t* req_trunk_start = meta + L.req_trunk_start;
  int32_t* req_prefix_off = meta + L.req_prefix_off;
  int32_t* req_first_q = meta + L.req_first_q;
  block_scan(R, [&](int j) { return P[j] - pl[j]; },
             [&](int j, long long e) { req_trunk_start[j] = static_cast<int32_t>(e); });
  long long prefix_total = block_scan(
      R, [&](int j) { return pl[j]; }, [&](int j, long long e) { req_prefix_off[j] = static_cast<int32_t>(e); });
  block_scan(R, [&](int j) { return n[j]; },
             [&](int j, long long e) { req_first_q[j] = static_cast<int32_t>(e); });
  for (int j = threadIdx.x; j < R; j += blockDim.x) {
    meta[L.req_trunk_len + j] = P[j];
    meta[L.req_prefix_len + j] = pl[j];
    meta[L.req_ckpt_pos + j] = ck[j];
    meta[L.req_n_q + j] = n[j];
    // trunk segment j
    meta[L.seg_start + j] = req_trunk_start[j];
    meta[L.seg_len + j] = P[j] - pl[j];
    meta[L.seg_pos0 + j] = pl[j];
    meta[L.seg_req + j] = j;
    meta[L.seg_branch + j] = 0;
    meta[L.seg_trunk_start + j] = req_trunk_start[j];
    meta[L.seg_trunk_len + j] = P[j] - pl[j];
    meta[L.seg_state_idx + j] = j;
  }
  if (threadIdx.x == 0) meta[H_PREFIX_TOTAL] = static_cast<int32_t>(prefix_total);
  __syncthreads();

  // ---- question segments -------------------------------------------------
  const int32_t t_trunk = static_cast<int32_t>(T_trunk);
  block_scan(Nq, [&](int i) { return ql[i]; }, [&](int i, long long e) {
    // request of question i: last j with first_q[j] <= i (requests without
    // questions share their successor's first_q and are skipped this way)
    int lo = 0, hi = R;  // answer in [lo, hi)
    while (hi - lo > 1) {
      int mid = (lo + hi) >> 1;
      if (req_first_q[mid] <= i) lo = mid; else hi = mid;
    }
    const int j = lo;
    const int s = R + i;
    const int32_t start = t_trunk + static_cast<int32_t>(e);
    meta[L.seg_start + s] = start;
    meta[L.seg_len + s] = ql[i];
    meta[L.seg_pos0 + s] = P[j];
    meta[L.seg_req + s] = j;
    meta[L.seg_branch + s] = i - req_first_q[j] + 1;
    meta[L.seg_trunk_start + s] = req_trunk_start[j];
    meta[L.seg_trunk_len + s] = P[j] - pl[j];
    meta[L.seg_state_idx + s] = j;
    meta[L.q_last + i] = start + ql[i] - 1;
  });
  __syncthreads();

  // ---- attention work list: tiles aligned to each segment start ----------
  const int nseg = R + Nq;
  int32_t* work_seg = meta + L.work_seg;
  int32_t* work_off = meta + L.work_off;
  const int32_t* seg_len = meta + L.seg_len;
  long long nwork = block_scan(nseg, [&](int s) { return (seg_len[s] + tile - 1) / tile; },
                               [&](int s, long long base) {
                                 const int c = (seg_len[s] + tile - 1) / tile;
                                 for (int u = 0; u < c; ++u) {
                                   work_seg[base + u] = s;
                                   work_off[base + u] = (c - 1 - u) * tile;
                                 }
                               });
  if (threadIdx.x == 0) meta[H_NWORK] = static_cast<int32_t>(nwork);
  __syncthreads();

  // ---- launch order: longest first ------------------------------------------
  // A work item's cost is its number of visible keys under full attention (the
  // position after its last query); items are launched in non-increasing cost,
  // ties in list order, so the long items start first and short ones fill the
  // tail.  Each item's result does not depend on the order.
  int32_t* order = meta + L.work_order;
  const int nw = static_cast<int>(nwork);
  __shared__ unsigned long long keys[kSortMax];
  if (nw > kSortMax) {
    for (int w = threadIdx.x; w < nw; w += blockDim.x) order[w] = w;
    return;
  }
  int np2 = 1;
  while (np2 < nw) np2 <<= 1;
  for (int w = threadIdx.x; w < np2; w += blockDim.x) {
    unsigned long long key = 0ull;
    if (w < nw) {
      const int s = work_seg[w], off = work_off[w];
      const int cost = meta[L.seg_pos0 + s] + off + min(tile, seg_len[s] - off);
      key = (static_cast<unsigned long long>(cost) << 32) | (0xFFFFFFFFu - static_cast<unsigned>(w));
    }
    keys[w] = key;
  }
  __syncthreads();
  // bitonic sort, descending
  for (int size = 2; size <= np2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < np2; i += blockDim.x) {
        const int jx = i ^ stride;
        if (jx > i) {
          const bool desc = (i & size) == 0;
          const unsigned long long a = keys[i], b = keys[jx];
          if (desc ? (a < b) : (a > b)) {
            keys[i] = b;
            keys[jx] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int w = threadIdx.x; w < nw; w += blockDim.x)
    order[w] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<unsigned>(keys[w] & 0xFFFFFFFFull));
}

// Per-token arrays: block b < nseg writes segment b's tokens; the last block
// writes the pad rows [T, T_cap).
__global__ void __launch_bounds__(256) meta_tokens_kernel(int32_t* __restrict__ meta, MetaLayout L) {
  const int b = blockIdx.x;
  const int nseg = meta[H_NSEG];
  if (b == L.max_seg) {
    const int T = meta[H_T];
    for (int x = T + threadIdx.x; x < L.T_cap; x += blockDim.x) {
      meta[L.tok_req + x] = -1;
      meta[L.tok_branch + x] = -1;
      meta[L.tok_pos + x] = -1;
    }
    return;
  }
  if (b >= nseg) return;
  const int32_t st = meta[L.seg_start + b], len = meta[L.seg_len + b];
  const int32_t j = meta[L.seg_req + b], c = meta[L.seg_branch + b], p0 = meta[L.seg_pos0 + b];
  for (int u = threadIdx.x; u < len; u += blockDim.x) {
    meta[L.tok_req + st + u] = j;
    meta[L.tok_branch + st + u] = c;
    meta[L.tok_pos + st + u] = p0 + u;
  }
}

// FORK_CHECKS: one block re-derives what the tables must satisfy and sets
// FORK_STATUS_CHECK on any mismatch.  Segments tile [0, T) in order, trunks
// first; each token's (request, branch, position) is its segment's; pad rows are
// -1; each work item lies inside its segment; question last rows end their
// segments.
__global__ void __launch_bounds__(1024) meta_check_kernel(int32_t* __restrict__ meta, MetaLayout L) {
  if (meta[H_VALID] == 0) return;
  const int R = meta[H_R], Nq = meta[H_NQ], T = meta[H_T], nseg = meta[H_NSEG], nwork = meta[H_NWORK];
  const int tile = meta[H_TILE];
  int bad = (nseg != R + Nq || T < 0 || T > L.T_cap || R > L.max_req || Nq > L.max_q || nwork > L.max_work ||
             tile < 1) ? 1 : 0;
  if (!bad) {
    for (int s = threadIdx.x; s < nseg; s += blockDim.x) {
      const int st = meta[L.seg_start + s], len = meta[L.seg_len + s], j = meta[L.seg_req + s];
      const int c = meta[L.seg_branch + s];
      const int end = s + 1 < nseg ? meta[L.seg_start + s + 1] : T;
      if (st < 0 || len < 0 || st + len != end || j < 0 || j >= R) { bad = 1; continue; }
      if ((s < R) != (c == 0) || (s >= R && len < 1)) bad = 1;
      if (meta[L.seg_trunk_start + s] != meta[L.seg_start + j] || meta[L.seg_trunk_len + s] != meta[L.seg_len + j] ||
          meta[L.seg_state_idx + s] != j)
        bad = 1;
      if (s >= R && meta[L.q_last + (s - R)] != st + len - 1) bad = 1;
    }
    if (nseg > 0 && meta[L.seg_start] != 0) bad = 1;
    for (int w = threadIdx.x; w < nwork; w += blockDim.x) {
      const int s = meta[L.work_seg + w], off = meta[L.work_off + w], o = meta[L.work_order + w];
      if (s < 0 || s >= nseg || off < 0 || off % tile != 0 || off >= meta[L.seg_len + s]) bad = 1;
      if (o < 0 || o >= nwork) bad = 1;
    }
    for (int x = threadIdx.x; x < L.T_cap; x += blockDim.x) {
      const int j = meta[L.tok_req + x], c = meta[L.tok_branch + x], t = meta[L.tok_pos + x];
      if (x >= T) {
        if (j != -1 || c != -1 || t != -1) bad = 1;
      } else if (j < 0 || j >= R || c < 0 || t < 0) {
        bad = 1;
      }
    }
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(meta + H_STATUS, FORK_STATUS_CHECK);
}

}  // namespace fork

using namespace fork;

extern "C" size_t fork_meta_bytes(int32_t T_cap, int32_t max_req, int32_t max_q) {
  if (!valid_caps(T_cap, max_req, max_q)) return 0;
  return static_cast<size_t>(meta_layout(T_cap, max_req, max_q).total) * 4;
}

extern "C" int fork_meta_init(fork_meta* m, void* d_buf, size_t bytes, int32_t T_cap,
                              int32_t max_req, int32_t max_q, int32_t tile_tokens) {
  if (!m) return FORK_EINVAL;
  fork_meta t;
  t.d_buf = d_buf;
  t.bytes = bytes;
  t.T_cap = T_cap;
  t.max_req = max_req;
  t.max_q = max_q;
  t.tile_tokens = tile_tokens;
  t.wait_us = 0;
  MetaLayout L;
  int rc = check_meta(&t, &L);
  if (rc != FORK_OK) return rc;
  *m = t;
  return FORK_OK;
}

extern "C" int fork_build_meta(const fork_meta* m, const int32_t* d_desc, int32_t R, int32_t Nq,
                               uint32_t flags, void* stream) {
  MetaLayout L;
  int rc = check_meta(m, &L);
  if (rc != FORK_OK) return rc;
  if (R < 0 || Nq < 0 || (!d_desc && (R > 0 || Nq > 0))) return FORK_EINVAL;
  if (R > m->max_req || Nq > m->max_q) return FORK_ECAPACITY;
  if ((rc = check_device()) != FORK_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* meta = static_cast<int32_t*>(m->d_buf);
  meta_tables_kernel<<<1, 1024, 0, s>>>(d_desc, R, Nq, 0, meta, L, m->tile_tokens);
  meta_tokens_kernel<<<L.max_seg + 1, 256, 0, s>>>(meta, L);
  if (flags & FORK_CHECKS) meta_check_kernel<<<1, 1024, 0, s>>>(meta, L);
  return cuda_rc(cudaGetLastError());
}

extern "C" size_t fork_desc_capacity_words(int32_t max_req, int32_t max_q) {
  if (max_req < 1 || max_req > (1 << 16) || max_q < 0 || max_q > (1 << 18)) return 0;
  return static_cast<size_t>(2) + 4 * static_cast<size_t>(max_req) + static_cast<size_t>(max_q);
}

extern "C" int fork_build_meta_dev(const fork_meta* m, const int32_t* d_desc, uint32_t flags, void* stream) {
  MetaLayout L;
  int rc = check_meta(m, &L);
  if (rc != FORK_OK) return rc;
  if (!d_desc) return FORK_EINVAL;
  if ((rc = check_device()) != FORK_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* meta = static_cast<int32_t*>(m->d_buf);
  meta_tables_kernel<<<1, 1024, 0, s>>>(d_desc, 0, 0, 1, meta, L, m->tile_tokens);
  meta_tokens_kernel<<<L.max_seg + 1, 256, 0, s>>>(meta, L);
  if (flags & FORK_CHECKS) meta_check_kernel<<<1, 1024, 0, s>>>(meta, L);
  return cuda_rc(cudaGetLastError());
}

extern "C" int fork_last_cuda_error(void) { return t_last_cuda_error; }

extern "C" int fork_read_status(const fork_meta* m, int32_t* h_status, void* stream) {
  MetaLayout L;
  int rc = check_meta(m, &L);
  if (rc != FORK_OK) return rc;
  if (!h_status) return FORK_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int32_t* meta = static_cast<const int32_t*>(m->d_buf);
  if (cuda_rc(cudaMemcpyAsync(h_status, meta + H_STATUS, sizeof(int32_t), cudaMemcpyDeviceToHost, s)) != FORK_OK)
    return FORK_ECUDA;
  return cuda_rc(cudaStreamSynchronize(s));
}
