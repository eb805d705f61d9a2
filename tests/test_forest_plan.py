"""The token-forest planner (host code of the C library, run here without a GPU)
against the forest's definition: node k's sequence is its ancestors' tokens, root
first, then its own (rainbus summary "未来方向" (2); the per-token rule of the
round, key visible iff it lies on the query's path at a position not after the
query's and, with a window, fewer than W positions before it).

Every table is derived again from the tree by brute force over rows and pairs:
positions, the rows each query sees, the levels and state indices, the leaves'
last rows, the work list's cover of the stream and its order.
"""
import numpy as np
import pytest

from tree_forked_hybrid_gb300 import build as B
from tree_forked_hybrid_gb300 import fork as F
from tree_forked_hybrid_gb300 import layout as LY

FORESTS = [
    # two trees (depth 3 and a leaf root); one-token leaf; lengths across tile boundaries
    ([-1, 0, 0, 1, 1, 1, 2, 2, 3, 3, -1], [30, 12, 8, 9, 4, 33, 6, 1, 5, 17, 45]),
    # a chain down to the deepest level allowed, an empty internal node, a wide last level
    ([-1, 0, 1, 2, 3, 4, 5, 6, 6, 6], [5, 3, 0, 7, 1, 2, 9, 4, 3, 6]),
    # an empty root, leaves at several depths, nodes listed out of depth order
    ([-1, 0, -1, 1, 2, 1, 4, 4, 0], [0, 6, 10, 3, 20, 2, 1, 8, 5]),
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    F.load()


def plan_of(parent, node_len, tile=16, T_cap=None, max_req=None, max_q=None):
    T = int(np.sum(node_len))
    T_cap = T_cap or T + 13
    max_req = max_req or len(parent)
    max_q = max_q or len(parent)
    img, plan = F.fork_forest_plan(T_cap, max_req, max_q, tile, parent, node_len)
    return LY.unpack(img, T_cap, max_req, max_q), plan, T_cap


def path_rows(parent, node_len, k):
    start = np.concatenate([[0], np.cumsum(node_len)[:-1]])
    chain = [k]
    while parent[chain[-1]] >= 0:
        chain.append(parent[chain[-1]])
    return np.concatenate([np.arange(start[a], start[a] + node_len[a]) for a in chain[::-1]]).astype(np.int64)


def node_of_row(node_len):
    return np.repeat(np.arange(len(node_len)), node_len)


@pytest.mark.parametrize("case", range(len(FORESTS)))
def test_header_positions_and_segments(case):
    parent, node_len = FORESTS[case]
    m, plan, T_cap = plan_of(parent, node_len)
    N, T = len(parent), int(np.sum(node_len))
    leaves = [k for k in range(N) if k not in parent]
    assert (m["R"], m["nseg"], m["Nq"], m["T"], m["valid"], m["forest"], m["status"]) == (
        N, N, len(leaves), T, 1, 1, 0)
    rows_node = node_of_row(node_len)
    for k in range(N):
        pr = path_rows(parent, node_len, k)
        own = pr[len(pr) - node_len[k]:]
        s = int(plan.state_index[k])
        # the node's own rows sit at the end of its path: positions continue along it
        assert np.array_equal(m["tok_pos"][own], np.arange(len(pr) - node_len[k], len(pr)))
        assert np.all(m["tok_req"][own] == s) and np.all(m["tok_branch"][own] == 0)
        assert m["seg_start"][s] == (own[0] if len(own) else np.sum(node_len[:k]))
        assert m["seg_len"][s] == node_len[k]
        assert m["seg_pos0"][s] == len(pr) - node_len[k] == m["req_prefix_len"][s]
        assert m["seg_state_idx"][s] == (plan.state_index[parent[k]] if parent[k] >= 0 else -1)
        assert m["req_ckpt_pos"][s] == -1
    assert np.all(m["tok_pos"][T:] == -1) and np.all(m["tok_req"][T:] == -1)
    assert np.array_equal(rows_node, np.repeat(np.arange(N), node_len))
    # the leaves' last rows, leaves in node order
    start = np.concatenate([[0], np.cumsum(node_len)[:-1]])
    assert np.array_equal(m["q_last"], [start[k] + node_len[k] - 1 for k in leaves])


@pytest.mark.parametrize("case", range(len(FORESTS)))
def test_levels_order_nodes_by_depth(case):
    parent, node_len = FORESTS[case]
    _, plan, _ = plan_of(parent, node_len)
    N = len(parent)

    def depth(k):
        d = 0
        while parent[k] >= 0:
            k, d = parent[k], d + 1
        return d

    depths = [depth(k) for k in range(N)]
    assert plan.levels == max(depths) + 1
    assert np.array_equal(np.sort(plan.state_index), np.arange(N))
    lf = plan.level_first
    assert lf[0] == 0 and lf[-1] == N and np.all(np.diff(lf) >= 1)
    for k in range(N):
        s = plan.state_index[k]
        assert lf[depths[k]] <= s < lf[depths[k] + 1]
        if parent[k] >= 0:  # the parent's state is complete one level earlier
            assert plan.state_index[parent[k]] < lf[depths[k]]
    for lv in range(plan.levels):  # node order inside a level
        nodes = sorted(range(N), key=lambda k: plan.state_index[k])[lf[lv]:lf[lv + 1]]
        assert nodes == sorted(nodes)


@pytest.mark.parametrize("case", range(len(FORESTS)))
@pytest.mark.parametrize("window", [0, 4, 11])
def test_visible_pairs_equal_the_path_definition(case, window):
    """The pairs the attention kernel's rule gives on these tables (parent chain through
    the state indices, then position and window) equal the pairs of the definition (the
    query's own path, positions not after it), and their count the closed form
    sum over queries of min(t + 1, W)."""
    parent, node_len = FORESTS[case]
    m, plan, _ = plan_of(parent, node_len)
    N, T = len(parent), int(np.sum(node_len))
    rows_node = node_of_row(node_len)
    pos = m["tok_pos"][:T]
    seg = m["tok_req"][:T]
    want = np.zeros((T, T), bool)
    for k in range(N):
        pr = path_rows(parent, node_len, k)
        for i in range(len(pr) - node_len[k], len(pr)):
            lo = max(0, i - window + 1) if window else 0
            want[pr[i], pr[lo:i + 1]] = True
    got = np.zeros((T, T), bool)
    for x in range(T):
        chain, s = set(), int(seg[x])
        for _ in range(F.FORK_FOREST_MAX_LEVELS):
            chain.add(s)
            s = int(m["seg_state_idx"][s])
            if s < 0:
                break
        assert s < 0, "parent chain longer than the levels"
        ok = np.isin(seg, list(chain)) & (pos <= pos[x])
        if window:
            ok &= pos[x] - pos < window
        got[x] = ok
    assert np.array_equal(got, want)
    W = window or 1 << 30
    assert got.sum() == sum(min(int(t) + 1, W) for t in pos)
    assert np.array_equal(rows_node, np.repeat(np.arange(N), node_len))


@pytest.mark.parametrize("case", range(len(FORESTS)))
@pytest.mark.parametrize("tile", [8, 16, 64])
def test_work_list_covers_the_stream_longest_first(case, tile):
    parent, node_len = FORESTS[case]
    m, _, _ = plan_of(parent, node_len, tile=tile)
    T = int(np.sum(node_len))
    cover = np.zeros(T, int)
    cost = []
    for w in range(m["n_work"]):
        s, off = int(m["work_seg"][w]), int(m["work_off"][w])
        st, ln = int(m["seg_start"][s]), int(m["seg_len"][s])
        assert off % tile == 0 and 0 <= off < ln
        n = min(tile, ln - off)
        cover[st + off:st + off + n] += 1
        cost.append(int(m["seg_pos0"][s]) + off + n)
    assert np.all(cover == 1)
    order = m["work_order"]
    assert np.array_equal(np.sort(order), np.arange(m["n_work"]))
    c = np.array(cost)[order]
    assert np.all(np.diff(c) <= 0)
    # ties keep list order
    for a, b in zip(order[:-1], order[1:]):
        if cost[a] == cost[b]:
            assert a < b


def test_planner_rejects_bad_forests():
    ok_p, ok_l = [-1, 0, 0], [4, 3, 2]
    plan_of(ok_p, ok_l)
    bad = [
        ([-1, 1, 0], [4, 3, 2], 1),        # parent after its child
        ([-1, -2, 0], [4, 3, 2], 1),       # parent index below -1
        ([-1, 0, 0], [4, -1, 2], 1),       # negative length
        ([-1, 0, 0], [4, 3, 0], 1),        # a leaf without tokens
    ]
    for parent, node_len, code in bad:
        with pytest.raises(F.ForkError) as e:
            F.fork_forest_plan(64, 8, 8, 16, parent, node_len)
        assert e.value.code == code
    with pytest.raises(F.ForkError) as e:  # more nodes than max_req
        F.fork_forest_plan(64, 2, 8, 16, ok_p, ok_l)
    assert e.value.code == 2
    with pytest.raises(F.ForkError) as e:  # more leaves than max_q
        F.fork_forest_plan(64, 8, 1, 16, ok_p, ok_l)
    assert e.value.code == 2
    with pytest.raises(F.ForkError) as e:  # more tokens than T_cap
        F.fork_forest_plan(8, 8, 8, 16, ok_p, ok_l)
    assert e.value.code == 2
    deep = list(range(-1, F.FORK_FOREST_MAX_DEPTH + 1))  # a chain of MAX_DEPTH + 2 nodes
    with pytest.raises(F.ForkError) as e:
        F.fork_forest_plan(64, 16, 8, 16, deep, [1] * len(deep))
    assert e.value.code == 2
    F.fork_forest_plan(64, 16, 8, 16, deep[:-1], [1] * (len(deep) - 1))  # the deepest allowed


def test_planner_equals_hand_derived_tables():
    """tests/golden/forest_cases.txt: tables worked out by hand from the forest rule."""
    from tests.golden_io import load_meta_cases
    cases = load_meta_cases("forest_cases.txt")
    assert cases
    for name, c in cases.items():
        parent, node_len = c["parent"], c["node_len"]
        N = parent.shape[0]
        T_cap, tile = int(c["T_cap"][0]), int(c["tile"][0])
        img, plan = F.fork_forest_plan(T_cap, N, N, tile, parent, node_len)
        m = LY.unpack(img, T_cap, N, N)
        assert m["T"] == int(c["T"][0]) and m["forest"] == 1, name
        assert plan.levels == int(c["levels"][0]), name
        assert plan.level_first.tolist() == c["level_first"].tolist(), name
        assert plan.state_index.tolist() == c["state_index"].tolist(), name
        for key in ("tok_req", "tok_pos", "seg_start", "seg_len", "seg_pos0", "seg_state_idx", "q_last",
                    "work_seg", "work_off", "work_order"):
            assert m[key][:c[key].shape[0]].tolist() == c[key].tolist(), (name, key)


def test_request_forest_shape():
    """The bench's forest: identical request trees, depth first, parents before children."""
    from tree_forked_hybrid_gb300 import workloads as wl
    parent, node_len = wl.request_forest(2, (4096, 512, 64), (4, 4))
    assert len(parent) == 2 * (1 + 4 + 16) and int(node_len.sum()) == 2 * (4096 + 4 * 512 + 16 * 64)
    assert all(-1 <= p < k for k, p in enumerate(parent))
    roots = [k for k in range(len(parent)) if parent[k] < 0]
    assert roots == [0, 21]
    for k in range(len(parent)):
        kids = [c for c in range(len(parent)) if parent[c] == k]
        depth = 0
        a = k
        while parent[a] >= 0:
            a, depth = parent[a], depth + 1
        assert len(kids) == (4 if depth < 2 else 0)
        assert node_len[k] == (4096, 512, 64)[depth]
    _, plan, _ = plan_of(parent, node_len, tile=64, T_cap=int(node_len.sum()))
    assert plan.levels == 3 and plan.level_first.tolist() == [0, 2, 10, 42]
