// Token forests in one flat stream: the host-side planner of the metadata.
//
// Source: rainbus summary "未来方向" (2) (a tree of draft tokens has the shape of
// the request tree and can run in the same flat stream as it); DFlash-TfM summary
// "GDN을 위한 롤백 없는 트리 검증" (the tree in topological order, the recurrence in
// its chunked form); onedev summary "무엇과 다른가" (the tree kept as metadata next
// to one unpadded stream; positions continue along a branch).
//
// A forest of N nodes, node k with parent[k] (-1 for a root, always an earlier
// node) and node_len[k] tokens stored node after node.  Node k's sequence is its
// ancestors' tokens, root first, then its own, so its first token has position
// pos0_k = sum of the ancestors' lengths.  The plan gives each node a segment whose
// index is its state index (nodes ordered by depth, then by node number, so that
// each depth is one contiguous run of indices, a launch of the recurrence), and
// fills the metadata tables that the kernels read:
//   - segment s: stream rows, length, pos0, state index of the parent (-1 for a
//     root), itself as request, branch 0 (trunk start/length = its own rows);
//   - request s: pos0 + length, pos0 as "prefix" (the recurrence starts from the
//     parent's state exactly when the node has tokens before it), no checkpoint;
//   - per token: segment, branch 0, position; pad rows -1;
//   - the last row of every leaf, leaves in node order (the readout's questions);
//   - the attention work list (tile_tokens-token tiles aligned to each segment's
//     first row, a segment's last tile first) and its order: non-increasing
//     visible keys (the position after the tile's last query), ties in list order.
// Plain host code: it runs (and is tested) without a GPU.
#include <algorithm>
#include <numeric>
#include <vector>

#include "fork_common.cuh"

using namespace fork;

extern "C" int fork_forest_plan(const fork_meta* m, const int32_t* parent, const int32_t* node_len, int32_t N,
                                int32_t* img, int32_t* plan) {
  MetaLayout L;
  int rc = check_meta(m, &L);
  if (rc != FORK_OK) return rc;
  if (!parent || !node_len || !img || !plan || N < 1) return FORK_EINVAL;
  // ---- validation ------------------------------------------------------------
  std::vector<char> has_child(N, 0);
  for (int k = 0; k < N; ++k) {
    if (parent[k] < -1 || parent[k] >= k || node_len[k] < 0) return FORK_EINVAL;
    if (parent[k] >= 0) has_child[parent[k]] = 1;
  }
  int n_leaves = 0;
  for (int k = 0; k < N; ++k) {
    if (has_child[k]) continue;
    if (node_len[k] < 1) return FORK_EINVAL;  // a leaf is a question: at least one token
    ++n_leaves;
  }
  if (N > L.max_req || n_leaves > L.max_q) return FORK_ECAPACITY;
  std::vector<int> depth(N);
  std::vector<int64_t> pos0(N), start(N);
  int64_t T = 0;
  int max_depth = 0;
  for (int k = 0; k < N; ++k) {
    const int p = parent[k];
    depth[k] = p < 0 ? 0 : depth[p] + 1;
    pos0[k] = p < 0 ? 0 : pos0[p] + node_len[p];
    start[k] = T;
    T += node_len[k];
    max_depth = std::max(max_depth, depth[k]);
  }
  if (T > L.T_cap || max_depth > FORK_FOREST_MAX_DEPTH) return FORK_ECAPACITY;

  // ---- state indices: by depth, then node number -----------------------------
  std::vector<int> node_of(N), seg_of(N);
  std::iota(node_of.begin(), node_of.end(), 0);
  std::stable_sort(node_of.begin(), node_of.end(), [&](int a, int b) { return depth[a] < depth[b]; });
  for (int s = 0; s < N; ++s) seg_of[node_of[s]] = s;

  // ---- tables ------------------------------------------------------------------
  std::fill(img, img + L.total, 0);
  const int tile = m->tile_tokens;
  for (int s = 0; s < N; ++s) {
    const int k = node_of[s];
    const int32_t st = static_cast<int32_t>(start[k]), len = node_len[k], p0 = static_cast<int32_t>(pos0[k]);
    img[L.seg_start + s] = st;
    img[L.seg_len + s] = len;
    img[L.seg_pos0 + s] = p0;
    img[L.seg_req + s] = s;
    img[L.seg_branch + s] = 0;
    img[L.seg_trunk_start + s] = st;
    img[L.seg_trunk_len + s] = len;
    img[L.seg_state_idx + s] = parent[k] < 0 ? -1 : seg_of[parent[k]];
    img[L.req_trunk_len + s] = p0 + len;
    img[L.req_prefix_len + s] = p0;
    img[L.req_prefix_off + s] = 0;
    img[L.req_ckpt_pos + s] = -1;
    img[L.req_trunk_start + s] = st;
    img[L.req_first_q + s] = 0;
    img[L.req_n_q + s] = 0;
    for (int u = 0; u < len; ++u) {
      img[L.tok_req + st + u] = s;
      img[L.tok_branch + st + u] = 0;
      img[L.tok_pos + st + u] = p0 + u;
    }
  }
  for (int64_t x = T; x < L.T_cap; ++x) {
    img[L.tok_req + x] = -1;
    img[L.tok_branch + x] = -1;
    img[L.tok_pos + x] = -1;
  }
  for (int k = 0, i = 0; k < N; ++k)
    if (!has_child[k]) img[L.q_last + i++] = static_cast<int32_t>(start[k] + node_len[k] - 1);

  // ---- attention work list and its order ------------------------------------------
  std::vector<int32_t> wseg, woff;
  for (int s = 0; s < N; ++s) {
    const int len = img[L.seg_len + s];
    const int c = (len + tile - 1) / tile;
    for (int u = 0; u < c; ++u) {
      wseg.push_back(s);
      woff.push_back((c - 1 - u) * tile);
    }
  }
  const int nw = static_cast<int>(wseg.size());
  if (nw > L.max_work) return FORK_ECAPACITY;
  std::vector<int64_t> cost(nw);
  for (int w = 0; w < nw; ++w) {
    const int s = wseg[w];
    cost[w] = static_cast<int64_t>(img[L.seg_pos0 + s]) + woff[w] + std::min(tile, img[L.seg_len + s] - woff[w]);
  }
  std::vector<int> order(nw);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return cost[a] > cost[b]; });
  for (int w = 0; w < nw; ++w) {
    img[L.work_seg + w] = wseg[w];
    img[L.work_off + w] = woff[w];
    img[L.work_order + w] = order[w];
  }

  // ---- header --------------------------------------------------------------------
  img[H_MAGIC] = kMagic;
  img[H_TCAP] = L.T_cap;
  img[H_MAXREQ] = L.max_req;
  img[H_MAXQ] = L.max_q;
  img[H_MAXSEG] = L.max_seg;
  img[H_MAXWORK] = L.max_work;
  img[H_R] = N;
  img[H_NQ] = n_leaves;
  img[H_T] = static_cast<int32_t>(T);
  img[H_NSEG] = N;
  img[H_TILE] = tile;
  img[H_NWORK] = nw;
  img[H_STATUS] = 0;
  img[H_PREFIX_TOTAL] = 0;
  img[H_VALID] = 1;
  img[H_FOREST] = 1;

  // ---- plan: levels and state indices ---------------------------------------------
  const int levels = max_depth + 1;
  plan[0] = levels;
  for (int l = 0, s = 0; l <= levels; ++l) {
    while (s < N && depth[node_of[s]] < l) ++s;
    plan[1 + l] = s;
  }
  for (int k = 0; k < N; ++k) plan[2 + FORK_FOREST_MAX_LEVELS + k] = seg_of[k];
  return FORK_OK;
}

extern "C" int fork_build_forest_meta(const fork_meta* m, const int32_t* parent, const int32_t* node_len, int32_t N,
                                      int32_t* img, int32_t* plan, void* stream) {
  int rc = fork_forest_plan(m, parent, node_len, N, img, plan);
  if (rc != FORK_OK) return rc;
  if ((rc = check_device()) != FORK_OK) return rc;
  const MetaLayout L = meta_layout(m->T_cap, m->max_req, m->max_q);
  return cuda_rc(cudaMemcpyAsync(m->d_buf, img, static_cast<size_t>(L.total) * 4, cudaMemcpyHostToDevice,
                                 static_cast<cudaStream_t>(stream)));
}
